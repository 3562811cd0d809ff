// moe_api.cu — the extern "C" entry points declared in include/moe.h: argument checks (before
// any CUDA call), device checks, workspace carving and the stream-ordered launches.
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int ok() {
    g_err[0] = '\0';
    return MOE_OK;
}

constexpr int kMaxE = 256, kMaxK = 8, kMaxDim = 65536;

bool dim_ok(int v) { return v >= 64 && v <= kMaxDim && v % 64 == 0; }

int check_shape(int T, int d, int f, int E, int k, bool need_f) {
    if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d must be >= 0", T);
    if (E < 1 || E > kMaxE) return fail(MOE_ERR_INVALID_ARG, "E = %d outside [1, %d]", E, kMaxE);
    if (k < 1 || k > E || k > kMaxK)
        return fail(MOE_ERR_INVALID_ARG, "top_k = %d outside [1, min(E=%d, %d)]", k, E, kMaxK);
    if (d != -1 && !dim_ok(d))
        return fail(MOE_ERR_INVALID_ARG, "d = %d must be a multiple of 64 in [64, %d]", d, kMaxDim);
    if (need_f && !dim_ok(f))
        return fail(MOE_ERR_INVALID_ARG, "f = %d must be a multiple of 64 in [64, %d]", f, kMaxDim);
    if (static_cast<long long>(T) * k >= (1ll << 31))
        return fail(MOE_ERR_INVALID_ARG, "T * top_k = %lld must be < 2^31", static_cast<long long>(T) * k);
    return MOE_OK;
}

struct DevInfo {
    int major = 0, minor = 0, sms = 0;
    bool init = false;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

// Current device must be compute capability 10.3; fills the SM count.
int check_device(int* num_sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(MOE_ERR_UNSUPPORTED, "device ordinal %d >= 64", dev);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DevInfo& di = g_dev[dev];
    if (!di.init) {
        if ((e = cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail(MOE_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        di.init = true;
    }
    if (di.major != 10 || di.minor != 3)
        return fail(MOE_ERR_UNSUPPORTED, "device %d is sm_%d%d; libmoe is built for sm_103a only", dev,
                    di.major, di.minor);
    *num_sms = di.sms;
    return MOE_OK;
}

int launched(cudaError_t e, const char* what) {
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
    return ok();
}

}  // namespace

// Default: every launch but the permute's.  Measured on GB300 (ms per layer, all five = 0.4197 at
// Mixtral T=32 against 0.4277 with none; but a programmatic permute launch costs the DeepSeek-
// shaped layer 0.09 ms: 2.545 with only that bit against 2.454 with none).
bool pdl_enabled(int kernel_bit) {
    static const int mask = [] {
        const char* v = std::getenv("MOE_PDL");
        return v ? std::atoi(v) : (kPdlRoute | kPdlGateUp | kPdlDown | kPdlCombine | kPdlQuant);
    }();
    return (mask & kernel_bit) != 0;
}

namespace {

// Experts with at most this many rows run the grouped GEMMs in the swapped orientation (weights
// as the UMMA M operand).  Per 64-deep K block the swapped MMAs read 32 KB of weights plus
// 256 B per row from shared memory against 48 KB for the normal 128x256 tile, so swapping pays
// below ~64 rows; measured on GB300 (Mixtral shape, T=512): 64 -> 0.574 ms/layer, 128 ->
// 0.589 ms.  MOE_GEMM_SWAP_MAX overrides it: 0 turns swapping off, values above 128 clamp to 128.
int swap_max_rows() {
    const char* v = std::getenv("MOE_GEMM_SWAP_MAX");
    int x = v ? std::atoi(v) : 64;
    return x < 0 ? 0 : (x > 128 ? 128 : x);
}

// Which grouped-GEMM kernel a layer shape runs on, per GEMM (kind 0 gate+up with N = f output
// columns, 1 down with N = d): 0 the 1-SM kernel (128-row tiles, experts with <= swap_max_rows()
// rows swapped), 1 the SM-pair kernel with 256-row tiles only, 2 the SM-pair kernel that also
// swaps small experts and the short remainders of large ones (and splits its CTA pairs between
// the two kinds of work where that pays).
//   * average expert >= 128 rows (M >= 128 E): SM pairs, so sibling M-tiles share one weight load;
//     gate+up in mode 2, the down GEMM in mode 1 (measured faster: Mixtral T=512 0.174 vs 0.185 ms,
//     T=4096 0.650 vs 0.665 — its 512-column swapped slots are coarser than its 256-column tiles);
//   * 32..127 rows per expert on average and at least 608 schedule slots (E x N/256 for gate+up,
//     E x N/512 for down: eight rounds over GB300's 76 SM pairs): mode 2 — many-expert layers mix
//     a few large experts, which pair tiles run faster, with many small ones, which stream swapped
//     (DeepSeek-V3 shape: gate+up 1.458 -> 1.197 ms, down 0.835 -> 0.764 ms); with fewer slots the
//     round-robin's last round runs mostly empty (a 32-expert layer of the same shape: gate+up
//     0.289 -> 0.340 ms);
//   * otherwise the 1-SM kernel.
// MOE_GEMM_2SM=0/1/2 overrides both GEMMs, MOE_GEMM_2SM_DOWN the down GEMM alone.
//
// The FP8 layer (fp8 = true) follows the same rules for gate+up (Mixtral shape, T=512: 0.196 ms on
// swapping pairs against 0.185 normal-only, but 0.183 against 0.209 with expert 0 drawing 40 % of
// the assignments; T=4096: 0.684 against 0.728; DeepSeek-V3 shape: 0.638 against 0.753 on single
// SMs); its down GEMM runs on normal-only pairs from 128 rows per expert and on single SMs below
// (DeepSeek-V3 shape: 0.499 ms against 0.576 on swapping pairs).
int use_pair(long long M, int E, int N, int kind, bool fp8 = false) {
    auto parse = [](const char* v) { return v[0] == '2' ? 2 : (v[0] == '1' ? 1 : 0); };
    if (kind == 1)
        if (const char* v = std::getenv("MOE_GEMM_2SM_DOWN")) return parse(v);
    if (const char* v = std::getenv("MOE_GEMM_2SM")) return parse(v);
    if (fp8 && kind == 1) return M >= 128ll * E ? 1 : 0;
    if (M >= 128ll * E) return kind == 1 ? 1 : 2;
    const int super_cols = kind == 0 ? 256 : 512;
    if (M >= 32ll * E && static_cast<long long>(E) * ((N + super_cols - 1) / super_cols) >= 608) return 2;
    return 0;
}

// Blockwise FP8: whether the gate+up GEMM quantises h in its epilogue (codes + 128-wide block
// scales; the separate quantisation launch goes) — when the experts hold more than 64 rows on
// average, so that most items are normal 128-row tiles.  The swapped items' epilogue shares each
// token's block maximum across four warps and costs more than the launch it saves (Mixtral shape,
// T=32, all items swapped: 0.253 vs 0.242 ms/layer; T=512 0.417 vs 0.430, T=4096 1.902 vs
// 1.944; DeepSeek-V3 shape, 64 rows per expert on average, 1.852 vs 1.846).
// MOE_FP8B_FUSE_H=0/1 overrides.
bool fp8b_fuse_h(long long M, int E) {
    if (const char* v = std::getenv("MOE_FP8B_FUSE_H")) return v[0] == '1';
    return M > 64ll * E;
}

// Swap threshold of the SM-pair kernel in mode 2: experts with at most this many rows run as one
// swapped chunk (further capped on the device at 64 or 128 rows by the shared-memory layout the
// kernel picks).  MOE_GEMM_PAIR_SWAP_MAX overrides (clamped to [0, 128]).
// Shared-memory layout of the swapping SM-pair kernel: 0 = chosen on the device from the row
// counts (default), 1 = layout A (six stages), 2 = layout B (five stages, 128-row chunks).
// MOE_GEMM_PAIR_LAYOUT overrides; a measurement knob.
int pair_layout() {
    const char* v = std::getenv("MOE_GEMM_PAIR_LAYOUT");
    return v ? (v[0] == 'A' || v[0] == '1' ? 1 : (v[0] == 'B' || v[0] == '2' ? 2 : 0)) : 0;
}

// Schedule of the swapping SM-pair kernel.  Default "auto" (1 << 21): the kernel splits its CTA
// pairs on the device between the normal tiles and the swapped chunks when both kinds carry much
// work and the tiles are tensor-bound (DeepSeek-V3 shape, gate+up: 1.394 -> 1.217 ms), else one
// round-robin over the slots in expert order.  MOE_GEMM_PAIR_SPLIT overrides: 0 = round-robin,
// P > 0 = P pairs on normal tiles, "mix" = round-robin over both kinds merged in proportion.
int pair_split() {
    const char* v = std::getenv("MOE_GEMM_PAIR_SPLIT");
    if (!v || v[0] == 'a') return 1 << 21;  // chosen on the device
    if (v[0] == 'm') return 1 << 20;        // proportional merge
    const int x = std::atoi(v);
    return x < 0 ? 0 : (x > 1000 ? 1000 : x);
}

int pair_swap_max_rows() {
    const char* v = std::getenv("MOE_GEMM_PAIR_SWAP_MAX");
    int x = v ? std::atoi(v) : 128;
    return x < 0 ? 0 : (x > 128 ? 128 : x);
}

// Whether moe_forward (and moe_forward_fp8) fold the combine into the down GEMM's epilogue instead of
// launching it (FoldArgs in common.cuh: per-(token, 64-column block) arrival counters, the last
// arrival sums the token's rows in slot order).  Off by default, MOE_FOLD_COMBINE=1 turns it on:
// measured slower at every bench workload (ms/layer, combine launch -> fold: Mixtral T=32 0.414 ->
// 0.428, T=512 0.506 -> 0.561, T=4096 1.94 -> 1.98, softmax-routed DeepSeek shape 2.11 -> 6.03,
// DeepSeek-V3 router 1.61 -> 4.52): a completing arrival sums the token's k rows in one thread,
// and at the end of the kernel those sums sit on its critical path.
bool fold_combine() {
    const char* v = std::getenv("MOE_FOLD_COMBINE");
    return v && v[0] == '1';
}

// Whether moe_forward's gate+up GEMM gathers its activation rows from x by src[] (the permute then
// writes no x_perm).  Off by default: measured slower than writing x_perm and reading it with TMA
// (Mixtral shape T=4096 2.81 vs 2.04 ms per layer, T=512 0.68 vs 0.53); MOE_GATHER=1 turns it on.
bool gather_rows() {
    const char* v = std::getenv("MOE_GATHER");
    return v && v[0] == '1';
}

// Whether moe_forward runs routing and the permutation as one launch (softmax router, E <= 32,
// T*E <= 8192: every block can afford to route all tokens itself).  MOE_FUSE_ROUTE_PERMUTE=0
// turns it off.
bool fuse_route_permute(int T, int E) {
    const char* v = std::getenv("MOE_FUSE_ROUTE_PERMUTE");
    if (v && v[0] == '0') return false;
    return route_permute_fusable(T, E);
}

// Failure-detection test hook, off unless the environment sets MOE_INJECT_STALL=1: the next
// grouped-GEMM launches (the stage calls' and the bf16 layer's) run on the 1-SM kernel with one
// pipeline stage armed for bytes that never arrive, so a bounded wait expires (~1 s), the kernel
// reports MOE_STATUS_WAIT_TIMEOUT in the status word, releases its tensor memory and returns.
// Nothing faults, traps or hangs.
int inject_stall() {
    const char* v = std::getenv("MOE_INJECT_STALL");
    return (v && v[0] == '1') ? 1 : 0;
}

// K slices for the down projection of a layer shape.  The down GEMM has d/256 N-tiles per M-tile.
// When that gives between one and two waves of work items on a 152-SM GB300, the last wave runs
// on a fraction of the SMs; splitting K in two evens it out (Mixtral shape, T=512: down GEMM
// 0.209 -> 0.179 ms).  Below one wave each item streams its own weight tile and the SMs in use
// already saturate HBM, and a split only adds partial-sum traffic (T=32: 0.138 -> 0.142 ms);
// above two waves the tail is small.  MOE_DOWN_KSPLIT overrides the choice.  The result never
// leaves a slice without K blocks.
// The FP8 layers (fp8 = true) have 128-deep K blocks; the blockwise one (blocks = true) always
// runs the 1-SM kernel.
int down_ksplit(int T, int d, int f, int E, int k, bool fp8 = false, bool blocks = false) {
    const long long M = static_cast<long long>(T) * k;
    const int num_kb = f / (fp8 ? 128 : 64);
    int S;
    if (const char* v = std::getenv("MOE_DOWN_KSPLIT")) {
        S = std::atoi(v);
    } else if (!blocks && use_pair(M, E, d, 1, fp8)) {
        S = 1;  // 256-row pair items: measured best unsplit (Mixtral T=512: 0.510 ms/layer vs 0.524 at 2)
    } else {
        const long long mtiles = (M + 127) / 128 + (M < E ? M : E);
        const long long items = mtiles * ((d + 255) / 256);
        S = (items >= 152 && items < 304) ? 2 : 1;
    }
    const int cap = num_kb < kMaxKSplit ? num_kb : kMaxKSplit;
    S = S < 1 ? 1 : (S > cap ? cap : S);
    const int per = (num_kb + S - 1) / S;
    return (num_kb + per - 1) / per;
}

// moe_forward's workspace: 256-byte aligned pieces in this order.
struct Layout {
    size_t status, idx, w, counts, offsets, src, dest, x_perm, h, y_perm, fold, total;
};

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

Layout layout(int T, int d, int f, int E, int k) {
    const size_t M = static_cast<size_t>(T) * k;
    Layout L;
    size_t o = 0;
    L.status = o; o += 256;
    L.idx = o; o = align256(o + M * 4);
    L.w = o; o = align256(o + M * 4);
    L.counts = o; o = align256(o + static_cast<size_t>(E) * 4);
    L.offsets = o; o = align256(o + static_cast<size_t>(E + 1) * 4);
    L.src = o; o = align256(o + M * 4);
    L.dest = o; o = align256(o + M * 4);
    L.x_perm = o; o = align256(o + M * d * 2);
    L.h = o; o = align256(o + M * f * 2);
    L.y_perm = o; o = align256(o + static_cast<size_t>(down_ksplit(T, d, f, E, k)) * M * d * 4);
    L.fold = o; o = align256(o + static_cast<size_t>(T) * (d / kFoldCols) * 4);  // combine-fold counters
    L.total = o;
    return L;
}

// The FP8 layer's workspace: the same first pieces, then x8 [M,d] codes, sx [M], h [M,f] bf16,
// h8 [M,f] codes, sh [M], y_perm.
struct Layout8 {
    size_t status, idx, w, counts, offsets, src, dest, x8, sx, h, h8, sh, y_perm, fold, total;
};

// blocks = true: the blockwise layer, whose sx and sh hold one scale per 128-wide block.
Layout8 layout_fp8(int T, int d, int f, int E, int k, bool blocks = false) {
    const size_t M = static_cast<size_t>(T) * k;
    const size_t nsx = blocks ? static_cast<size_t>(d / 128) : 1, nsh = blocks ? static_cast<size_t>(f / 128) : 1;
    Layout8 L;
    size_t o = 0;
    L.status = o; o += 256;
    L.idx = o; o = align256(o + M * 4);
    L.w = o; o = align256(o + M * 4);
    L.counts = o; o = align256(o + static_cast<size_t>(E) * 4);
    L.offsets = o; o = align256(o + static_cast<size_t>(E + 1) * 4);
    L.src = o; o = align256(o + M * 4);
    L.dest = o; o = align256(o + M * 4);
    L.x8 = o; o = align256(o + M * d);
    L.sx = o; o = align256(o + M * nsx * 4);
    L.h = o; o = align256(o + M * f * 2);
    L.h8 = o; o = align256(o + M * f);
    L.sh = o; o = align256(o + M * nsh * 4);
    L.y_perm = o; o = align256(o + static_cast<size_t>(down_ksplit(T, d, f, E, k, true, blocks)) * M * d * 4);
    L.fold = o; o = align256(o + static_cast<size_t>(T) * (d / kFoldCols) * 4);  // combine-fold counters
    L.total = o;
    return L;
}

template <class P>
P* at(void* base, size_t off) {
    return reinterpret_cast<P*>(static_cast<char*>(base) + off);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The router of a layer: the softmax top-k router when `grouped` is false, else DeepSeek-V3's
// (sigmoid affinity, selection bias, group-limited top-k, scaled weights).
struct Router {
    bool grouped = false;
    const float* bias = nullptr;
    int n_group = 1, topk_group = 1;
    float scale = 1.0f;
};

int check_router(const Router& r, int E, int k, const char* name) {
    if (!r.grouped) return MOE_OK;
    if (!r.bias) return fail(MOE_ERR_INVALID_ARG, "%s: null bias", name);
    if (r.n_group < 1 || r.n_group > 32 || E % r.n_group != 0)
        return fail(MOE_ERR_INVALID_ARG, "%s: n_group = %d must divide E = %d and lie in [1, 32]", name, r.n_group, E);
    if (r.topk_group < 1 || r.topk_group > r.n_group)
        return fail(MOE_ERR_INVALID_ARG, "%s: topk_group = %d outside [1, n_group = %d]", name, r.topk_group,
                    r.n_group);
    if (k > r.topk_group * (E / r.n_group))
        return fail(MOE_ERR_INVALID_ARG, "%s: top_k = %d exceeds the %d experts of the kept groups", name, k,
                    r.topk_group * (E / r.n_group));
    if (!(r.scale > 0.0f) || r.scale > 3.0e38f)
        return fail(MOE_ERR_INVALID_ARG, "%s: scale must be a positive finite number", name);
    return MOE_OK;
}

int run_layer(const void* x, const float* logits, const void* wgu, const void* wd, int T, int d, int f,
              int E, int k, void* out, void* ws, int num_sms, cudaStream_t s, const Router& router = Router()) {
    const Layout L = layout(T, d, f, E, k);
    int32_t* status = at<int32_t>(ws, L.status);
    int32_t* idx = at<int32_t>(ws, L.idx);
    float* w = at<float>(ws, L.w);
    int32_t* counts = at<int32_t>(ws, L.counts);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* src = at<int32_t>(ws, L.src);
    int32_t* dest = at<int32_t>(ws, L.dest);
    auto* x_perm = at<__nv_bfloat16>(ws, L.x_perm);
    auto* h = at<__nv_bfloat16>(ws, L.h);
    float* y = at<float>(ws, L.y_perm);
    const int M = T * k;
    cudaError_t e;
    const bool gather = gather_rows();
    __nv_bfloat16* xp = gather ? nullptr : x_perm;  // no x_perm when the GEMM gathers
    int32_t* fold_cnt = fold_combine() ? at<int32_t>(ws, L.fold) : nullptr;  // zeroed by the permute
    const int fold_nblk = d / kFoldCols;
    if (!router.grouped && fuse_route_permute(T, E)) {
        if ((e = launch_route_permute(logits, static_cast<const __nv_bfloat16*>(x), T, d, E, k, idx, w, counts,
                                      offsets, src, dest, xp, status, num_sms, s, nullptr, nullptr, fold_cnt,
                                      fold_nblk)) != cudaSuccess)
            return launched(e, "route+permute");
    } else {
        e = router.grouped ? launch_route_grouped(logits, router.bias, T, E, k, router.n_group, router.topk_group,
                                                  router.scale, idx, w, status, s)
                           : launch_route(logits, T, E, k, idx, w, status, s);
        if (e != cudaSuccess) return launched(e, "route");
        if ((e = launch_permute(idx, static_cast<const __nv_bfloat16*>(x), T, d, E, k, counts, offsets, src,
                                dest, xp, status, num_sms, s, nullptr, nullptr, fold_cnt, fold_nblk)) != cudaSuccess)
            return launched(e, "permute");
    }
    const char* why = "";
    const int swap_max = swap_max_rows(), ksplit = down_ksplit(T, d, f, E, k);
    GemmArgs g1{gather ? x : x_perm, wgu, offsets, M, d, f, E, h, status, 1, swap_max, use_pair(M, E, f, 0),
                pair_swap_max_rows(), pair_layout(), pair_split()};
    if (gather) {
        g1.gather_src = src;
        g1.gather_T = T;
    }
    g1.inject_stall = inject_stall();  // failure-detection test hook, off unless MOE_INJECT_STALL=1
    if ((e = launch_grouped_gemm(0, g1, num_sms, s, &why)) != cudaSuccess)
        return fail(MOE_ERR_CUDA, "gate+up GEMM: %s (%s)", why, cudaGetErrorString(e));
    GemmArgs g2{h, wd, offsets, M, f, d, E, y, status, ksplit, swap_max, use_pair(M, E, d, 1), pair_swap_max_rows(),
                pair_layout(), pair_split()};
    g2.inject_stall = g1.inject_stall;
    if (fold_cnt) g2.fold = FoldArgs{fold_cnt, src, dest, w, static_cast<__nv_bfloat16*>(out), T, k};
    if ((e = launch_grouped_gemm(1, g2, num_sms, s, &why)) != cudaSuccess)
        return fail(MOE_ERR_CUDA, "down GEMM: %s (%s)", why, cudaGetErrorString(e));
    if (!fold_cnt &&
        (e = launch_combine(y, w, dest, T, d, k, ksplit, static_cast<__nv_bfloat16*>(out), status, s)) != cudaSuccess)
        return launched(e, "combine");
    return ok();
}

// The FP8 layers.  Per-row / per-channel scales (blocks = false): route (+ permute writing the x
// rows quantised), gate+up FP8 GEMM (+ SwiGLU, bf16 h), h quantised per row, down FP8 GEMM,
// combine.  Blockwise scales (blocks = true): the permutation computes indices only and x rows are
// gathered by src and quantised in 128-wide blocks by their own launch; the GEMMs are the
// blockwise kernel's.
int run_layer_fp8(const void* x, const float* logits, const void* wgu8, const float* sgu, const void* wd8,
                  const float* sd, int T, int d, int f, int E, int k, void* out, void* ws, int num_sms,
                  cudaStream_t s, bool blocks, const Router& router = Router()) {
    const Layout8 L = layout_fp8(T, d, f, E, k, blocks);
    int32_t* status = at<int32_t>(ws, L.status);
    int32_t* idx = at<int32_t>(ws, L.idx);
    float* w = at<float>(ws, L.w);
    int32_t* counts = at<int32_t>(ws, L.counts);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* src = at<int32_t>(ws, L.src);
    int32_t* dest = at<int32_t>(ws, L.dest);
    uint8_t* x8 = at<uint8_t>(ws, L.x8);
    float* sx = at<float>(ws, L.sx);
    auto* h = at<__nv_bfloat16>(ws, L.h);
    uint8_t* h8 = at<uint8_t>(ws, L.h8);
    float* sh = at<float>(ws, L.sh);
    float* y = at<float>(ws, L.y_perm);
    const int M = T * k;
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    uint8_t* perm_x8 = blocks ? nullptr : x8;  // per-row scales: the permutation quantises x itself
    float* perm_sx = blocks ? nullptr : sx;
    // The combine folds into the per-row-scaled down GEMM (the blockwise kernel has no fold).
    int32_t* fold_cnt = (!blocks && fold_combine()) ? at<int32_t>(ws, L.fold) : nullptr;
    const int fold_nblk = d / kFoldCols;
    cudaError_t e;
    if (!router.grouped && fuse_route_permute(T, E)) {
        if ((e = launch_route_permute(logits, xb, T, d, E, k, idx, w, counts, offsets, src, dest, nullptr, status,
                                      num_sms, s, perm_x8, perm_sx, fold_cnt, fold_nblk)) != cudaSuccess)
            return launched(e, "route+permute");
    } else {
        e = router.grouped ? launch_route_grouped(logits, router.bias, T, E, k, router.n_group, router.topk_group,
                                                  router.scale, idx, w, status, s)
                           : launch_route(logits, T, E, k, idx, w, status, s);
        if (e != cudaSuccess) return launched(e, "route");
        if ((e = launch_permute(idx, xb, T, d, E, k, counts, offsets, src, dest, nullptr, status, num_sms, s, perm_x8,
                                perm_sx, fold_cnt, fold_nblk)) != cudaSuccess)
            return launched(e, "permute");
    }
    if (blocks && (e = launch_quantize_rows_fp8b(xb, src, M, d, T, x8, sx, status, s)) != cudaSuccess)
        return launched(e, "quantize x");
    auto gemm = [&](int kind, GemmArgs& g, const char* what) -> int {
        const char* why = "";
        const cudaError_t ge = blocks ? launch_grouped_gemm_fp8b(kind, g, num_sms, s, &why)
                                      : launch_grouped_gemm(kind, g, num_sms, s, &why);
        return ge == cudaSuccess ? MOE_OK : fail(MOE_ERR_CUDA, "%s: %s (%s)", what, why, cudaGetErrorString(ge));
    };
    const int ksplit = down_ksplit(T, d, f, E, k, true, blocks);
    // Blockwise, by fp8b_fuse_h: the gate+up GEMM writes h's codes and 128-wide block scales itself
    // (h in bf16 never exists).  Otherwise, and always for per-row scales (which need the whole
    // row), h is quantised by a launch of its own.
    const bool fuse_h = blocks && fp8b_fuse_h(M, E);
    GemmArgs g1{x8, wgu8, offsets, M, d, f, E, fuse_h ? static_cast<void*>(h8) : h, status, 1, swap_max_rows(),
                blocks ? 0 : use_pair(M, E, f, 0, true), pair_swap_max_rows(), pair_layout(), pair_split()};
    g1.fp8 = true;
    g1.fp8_blocks = blocks;
    g1.a_scale = sx;
    g1.b_scale = sgu;
    if (fuse_h) g1.h_scale = sh;
    int rc = gemm(0, g1, blocks ? "blockwise FP8 gate+up GEMM" : "FP8 gate+up GEMM");
    if (rc) return rc;
    if (!fuse_h) {
        e = blocks ? launch_quantize_rows_fp8b(h, nullptr, M, f, M, h8, sh, status, s)
                   : launch_quantize_rows_fp8(h, nullptr, M, f, M, h8, sh, status, s);
        if (e != cudaSuccess) return launched(e, "quantize h");
    }
    GemmArgs g2{h8, wd8, offsets, M, f, d, E, y, status, ksplit, swap_max_rows(),
                blocks ? 0 : use_pair(M, E, d, 1, true), pair_swap_max_rows(), pair_layout(), pair_split()};
    g2.fp8 = true;
    g2.fp8_blocks = blocks;
    g2.a_scale = sh;
    g2.b_scale = sd;
    if (fold_cnt) g2.fold = FoldArgs{fold_cnt, src, dest, w, static_cast<__nv_bfloat16*>(out), T, k};
    if ((rc = gemm(1, g2, blocks ? "blockwise FP8 down GEMM" : "FP8 down GEMM"))) return rc;
    if (!fold_cnt &&
        (e = launch_combine(y, w, dest, T, d, k, ksplit, static_cast<__nv_bfloat16*>(out), status, s)) != cudaSuccess)
        return launched(e, "combine");
    return ok();
}

bool dim8_ok(int v) { return v % 128 == 0; }

int check_shape_fp8(int T, int d, int f, int E, int k, const char* name) {
    int rc = check_shape(T, d, f, E, k, true);
    if (rc) return rc;
    if (!dim8_ok(d) || !dim8_ok(f))
        return fail(MOE_ERR_INVALID_ARG, "%s: d = %d and f = %d must be multiples of 128 (FP8 K blocks)", name, d, f);
    return MOE_OK;
}

}  // namespace
}  // namespace moe

// Scratch of moe_forward_noalloc: one fixed device array per GPU, never allocated at run time.
static __device__ __align__(256) unsigned char moe_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

namespace moe {
namespace {

std::mutex g_noalloc_mu;
constexpr int kNoallocMaxDevices = 64;
// Per device: the array's device address and the CUDA context it was looked up in.  A context
// destroyed and created again (cudaDeviceReset, or the primary context released and retained)
// loads the module again, and the array can move; the address is then looked up afresh.
void* g_noalloc_ptr[kNoallocMaxDevices] = {};
void* g_noalloc_ctx[kNoallocMaxDevices] = {};

// The current thread's CUDA context (driver cuCtxGetCurrent, reached through the runtime's
// entry-point query so that the library needs no link against libcuda).
int current_context(void** ctx) {
    using GetCurrent = int (*)(void**);
    static GetCurrent fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<GetCurrent>(p);
    });
    *ctx = nullptr;
    if (!fn) return fail(MOE_ERR_CUDA, "moe_forward_noalloc: driver entry point cuCtxGetCurrent not found");
    if (fn(ctx) != 0 || *ctx == nullptr)
        return fail(MOE_ERR_CUDA, "moe_forward_noalloc: no current CUDA context");
    return MOE_OK;
}

// Device address of moe_noalloc_scratch on device `dev` (current), looked up with that device
// current the first time a context of it is seen.  In host code the array's name is only a
// host-side handle, never a device address.
int noalloc_scratch(int dev, void** out) {
    if (dev < 0 || dev >= kNoallocMaxDevices)
        return fail(MOE_ERR_UNSUPPORTED, "moe_forward_noalloc: device ordinal %d is beyond the %d this library tracks",
                    dev, kNoallocMaxDevices);
    void* ctx = nullptr;
    int rc = current_context(&ctx);
    if (rc) return rc;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr || g_noalloc_ctx[dev] != ctx) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, moe_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return fail(MOE_ERR_CUDA, "moe_forward_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        g_noalloc_ptr[dev] = p;
        g_noalloc_ctx[dev] = ctx;
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

// Null checks of the *_host_batches calls' per-batch host pointers.
static int check_host_batches(const char* name, const void* const* x_hosts, const float* const* logits_hosts,
                              void* const* out_hosts, int n_batches) {
    if (!x_hosts || !logits_hosts || !out_hosts) return fail(MOE_ERR_INVALID_ARG, "%s: null pointer", name);
    for (int b = 0; b < n_batches; ++b)
        if (!x_hosts[b] || !logits_hosts[b] || !out_hosts[b])
            return fail(MOE_ERR_INVALID_ARG, "%s: null host pointer for batch %d", name, b);
    return MOE_OK;
}

// The copy/compute pipeline of the *_host_batches calls (arguments already checked): two staging
// slots (x, out, logits, as moe_forward_host lays them out) after the layer's `need` bytes of
// workspace; batch b's inputs go to slot b & 1 on `si` once the layer of batch b-2 has read it,
// its layer runs on `s` (run(x_dev, logits_dev, out_dev)) once they have landed and batch b-2's
// output has left the slot, and its output goes back on `so`.
template <typename Run>
static int run_host_batches(const char* name, const void* const* x_hosts, const float* const* logits_hosts,
                            void* const* out_hosts, int n_batches, int T, int d, int E, size_t need, void* workspace,
                            cudaStream_t s, cudaStream_t si, cudaStream_t so, Run run) {
    const size_t stage = moe_host_staging_size(T, d, E);
    const size_t xb = static_cast<size_t>(T) * d * 2, lb = static_cast<size_t>(T) * E * 4;
    void* x_dev[2];
    void* out_dev[2];
    float* logits_dev[2];
    for (int k = 0; k < 2; ++k) {
        const size_t base = need + k * stage;
        x_dev[k] = at<char>(workspace, base);
        out_dev[k] = at<char>(workspace, base + align256(xb));
        logits_dev[k] = at<float>(workspace, base + 2 * align256(xb));
    }
    // Events: start (prior work on `s`), and per slot: inputs landed, layer done, output read.
    cudaEvent_t ev[7] = {};
    cudaError_t e = cudaSuccess;
    for (int k = 0; k < 7 && e == cudaSuccess; ++k) e = cudaEventCreateWithFlags(&ev[k], cudaEventDisableTiming);
    cudaEvent_t start = ev[0], in_ready[2] = {ev[1], ev[2]}, layer_done[2] = {ev[3], ev[4]},
                out_done[2] = {ev[5], ev[6]};
    auto cleanup = [&]() {
        for (int k = 0; k < 7; ++k)
            if (ev[k]) cudaEventDestroy(ev[k]);  // released once the recorded work completes
    };
    if (e != cudaSuccess) {
        cleanup();
        return fail(MOE_ERR_CUDA, "%s: event creation: %s", name, cudaGetErrorString(e));
    }
    // Everything below is ordered after the work already enqueued on `s` (which may still be
    // using the staging slots or the layer's workspace).
    if ((e = cudaEventRecord(start, s)) != cudaSuccess || (e = cudaStreamWaitEvent(si, start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(so, start, 0)) != cudaSuccess) {
        cleanup();
        return fail(MOE_ERR_CUDA, "%s: stream ordering: %s", name, cudaGetErrorString(e));
    }
    int rc = MOE_OK;
    for (int b = 0; b < n_batches && e == cudaSuccess && rc == MOE_OK; ++b) {
        const int k = b & 1;
        if (b >= 2 && (e = cudaStreamWaitEvent(si, layer_done[k], 0)) != cudaSuccess) break;
        if ((e = cudaMemcpyAsync(x_dev[k], x_hosts[b], xb, cudaMemcpyHostToDevice, si)) != cudaSuccess ||
            (e = cudaMemcpyAsync(logits_dev[k], logits_hosts[b], lb, cudaMemcpyHostToDevice, si)) != cudaSuccess ||
            (e = cudaEventRecord(in_ready[k], si)) != cudaSuccess)
            break;
        if ((e = cudaStreamWaitEvent(s, in_ready[k], 0)) != cudaSuccess) break;
        if (b >= 2 && (e = cudaStreamWaitEvent(s, out_done[k], 0)) != cudaSuccess) break;
        if ((rc = run(x_dev[k], logits_dev[k], out_dev[k])) != MOE_OK) break;
        if ((e = cudaEventRecord(layer_done[k], s)) != cudaSuccess) break;
        if ((e = cudaStreamWaitEvent(so, layer_done[k], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(out_hosts[b], out_dev[k], xb, cudaMemcpyDeviceToHost, so)) != cudaSuccess ||
            (e = cudaEventRecord(out_done[k], so)) != cudaSuccess)
            break;
    }
    // `s` completes only after the last copy back (the copies on `so` run in order).
    if (e == cudaSuccess && rc == MOE_OK) e = cudaStreamWaitEvent(s, out_done[(n_batches - 1) & 1], 0);
    cleanup();
    if (rc != MOE_OK) return rc;
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", name, cudaGetErrorString(e));
    return ok();
}

extern "C" {

int moe_version(void) { return 100; }

int moe_forward_launch_count(int T, int E, int top_k) {
    if (check_shape(T, -1, 0, E, top_k, false) != MOE_OK) return -1;
    if (T == 0) return 0;
    return (fuse_route_permute(T, E) ? 4 : 5) - (fold_combine() ? 1 : 0);
}

const char* moe_last_error_string(void) { return g_err; }

size_t moe_workspace_size(int T, int d, int f, int E, int top_k) {
    if (check_shape(T, d, f, E, top_k, true) != MOE_OK) return 0;
    return layout(T, d, f, E, top_k).total;
}

int moe_workspace_layout(int T, int d, int f, int E, int top_k, size_t* offsets_out) {
    int rc = check_shape(T, d, f, E, top_k, true);
    if (rc) return rc;
    if (!offsets_out) return fail(MOE_ERR_INVALID_ARG, "moe_workspace_layout: null pointer");
    const Layout L = layout(T, d, f, E, top_k);
    const size_t v[11] = {L.status, L.idx, L.w, L.counts, L.offsets, L.src, L.dest, L.x_perm, L.h, L.y_perm, L.total};
    for (int i = 0; i < 11; ++i) offsets_out[i] = v[i];
    return ok();
}

int moe_gemm_pair_mode(int T, int d, int f, int E, int top_k, int kind) {
    if (check_shape(T, d, f, E, top_k, true) != MOE_OK || (kind != 0 && kind != 1)) return -1;
    return use_pair(static_cast<long long>(T) * top_k, E, kind == 0 ? f : d, kind);
}

int moe_down_ksplit(int T, int d, int f, int E, int top_k) {
    if (check_shape(T, d, f, E, top_k, true) != MOE_OK) return 0;
    return down_ksplit(T, d, f, E, top_k);
}

size_t moe_host_staging_size(int T, int d, int E) {
    if (T < 0 || d < 1 || E < 1) return 0;
    return align256(static_cast<size_t>(T) * d * 2) * 2 + align256(static_cast<size_t>(T) * E * 4);
}

int moe_route(const float* logits, int T, int E, int top_k, int32_t* idx, float* w, moe_stream_t stream) {
    int rc = check_shape(T, -1, 0, E, top_k, false);
    if (rc) return rc;
    if (T == 0) return ok();
    if (!logits || !idx || !w) return fail(MOE_ERR_INVALID_ARG, "moe_route: null pointer");
    int sms;
    if ((rc = check_device(&sms))) return rc;
    return launched(launch_route(logits, T, E, top_k, idx, w, nullptr, static_cast<cudaStream_t>(stream)),
                    "route");
}

int moe_route_grouped(const float* logits, const float* bias, int T, int E, int top_k, int n_group,
                      int topk_group, float scale, int32_t* idx, float* w, moe_stream_t stream) {
    int rc = check_shape(T, -1, 0, E, top_k, false);
    if (rc) return rc;
    Router r;
    r.grouped = true;
    r.bias = bias;
    r.n_group = n_group;
    r.topk_group = topk_group;
    r.scale = scale;
    if ((rc = check_router(r, E, top_k, "moe_route_grouped"))) return rc;
    if (T == 0) return ok();
    if (!logits || !idx || !w) return fail(MOE_ERR_INVALID_ARG, "moe_route_grouped: null pointer");
    int sms;
    if ((rc = check_device(&sms))) return rc;
    return launched(launch_route_grouped(logits, bias, T, E, top_k, n_group, topk_group, scale, idx, w, nullptr,
                                         static_cast<cudaStream_t>(stream)),
                    "route_grouped");
}

int moe_permute(const int32_t* idx, const void* x, int T, int d, int E, int top_k, int32_t* counts,
                int32_t* offsets, int32_t* src, int32_t* dest, void* x_perm, int32_t* status,
                moe_stream_t stream) {
    int rc = check_shape(T, d, 0, E, top_k, false);
    if (rc) return rc;
    if (T == 0) return ok();
    if (!idx || !x || !counts || !offsets || !src || !dest)
        return fail(MOE_ERR_INVALID_ARG, "moe_permute: null pointer");
    if (!aligned16(x) || (x_perm && !aligned16(x_perm)))
        return fail(MOE_ERR_INVALID_ARG, "moe_permute: x and x_perm must be 16-byte aligned");
    int sms;
    if ((rc = check_device(&sms))) return rc;
    return launched(launch_permute(idx, static_cast<const __nv_bfloat16*>(x), T, d, E, top_k, counts,
                                   offsets, src, dest, static_cast<__nv_bfloat16*>(x_perm), status, sms,
                                   static_cast<cudaStream_t>(stream)),
                    "permute");
}

static int gemm_entry(int kind, const void* A, const void* B, const int32_t* offsets, int M, int d, int f,
                      int E, int ksplit, void* out, int32_t* status, moe_stream_t stream, const char* name,
                      const int32_t* gather_src = nullptr, int gather_T = 0) {
    int rc = check_shape(0, d, f, E, 1, true);
    if (rc) return rc;
    if (M < 0) return fail(MOE_ERR_INVALID_ARG, "%s: M = %d must be >= 0", name, M);
    if (ksplit < 1 || ksplit > kMaxKSplit)
        return fail(MOE_ERR_INVALID_ARG, "%s: ksplit = %d outside [1, %d]", name, ksplit, kMaxKSplit);
    if (M == 0) return ok();
    if (!A || !B || !offsets || !out) return fail(MOE_ERR_INVALID_ARG, "%s: null pointer", name);
    if (!aligned16(A) || !aligned16(B) || !aligned16(out))
        return fail(MOE_ERR_INVALID_ARG, "%s: operands must be 16-byte aligned", name);
    int sms;
    if ((rc = check_device(&sms))) return rc;
    const int pair = use_pair(M, E, kind == 0 ? f : d, kind);
    GemmArgs g = kind == 0 ? GemmArgs{A, B, offsets, M, d, f, E, out, status, 1, swap_max_rows(), pair}
                           : GemmArgs{A, B, offsets, M, f, d, E, out, status, ksplit, swap_max_rows(), pair};
    g.pair_swap_max = pair_swap_max_rows();
    g.pair_layout = pair_layout();
    g.pair_split = pair_split();
    g.inject_stall = inject_stall();
    g.gather_src = gather_src;
    g.gather_T = gather_T;
    const char* why = "";
    cudaError_t e = launch_grouped_gemm(kind, g, sms, static_cast<cudaStream_t>(stream), &why);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s (%s)", name, why, cudaGetErrorString(e));
    return ok();
}

int moe_grouped_gemm_gateup_swiglu(const void* x_perm, const void* w_gate_up, const int32_t* offsets, int M,
                                   int d, int f, int E, void* h, int32_t* status, moe_stream_t stream) {
    return gemm_entry(0, x_perm, w_gate_up, offsets, M, d, f, E, 1, h, status, stream,
                      "moe_grouped_gemm_gateup_swiglu");
}

int moe_grouped_gemm_gateup_swiglu_gather(const void* x, const int32_t* src, int T, const void* w_gate_up,
                                          const int32_t* offsets, int M, int d, int f, int E, void* h,
                                          int32_t* status, moe_stream_t stream) {
    if (T < 0) return fail(MOE_ERR_INVALID_ARG, "moe_grouped_gemm_gateup_swiglu_gather: T = %d must be >= 0", T);
    if (M > 0 && (!src || T == 0))
        return fail(MOE_ERR_INVALID_ARG, "moe_grouped_gemm_gateup_swiglu_gather: null src or empty x");
    return gemm_entry(0, x, w_gate_up, offsets, M, d, f, E, 1, h, status, stream,
                      "moe_grouped_gemm_gateup_swiglu_gather", src, T);
}

int moe_grouped_gemm_down(const void* h, const void* w_down, const int32_t* offsets, int M, int d, int f,
                          int E, int ksplit, float* y_perm, int32_t* status, moe_stream_t stream) {
    return gemm_entry(1, h, w_down, offsets, M, d, f, E, ksplit, y_perm, status, stream, "moe_grouped_gemm_down");
}

int moe_combine(const float* y_perm, const float* w, const int32_t* dest, int T, int d, int top_k, int ksplit,
                void* out, int32_t* status, moe_stream_t stream) {
    int rc = check_shape(T, d, 0, top_k, top_k, false);
    if (rc) return rc;
    if (T == 0) return ok();
    if (!y_perm || !w || !dest || !out) return fail(MOE_ERR_INVALID_ARG, "moe_combine: null pointer");
    if (ksplit < 1 || ksplit > kMaxKSplit)
        return fail(MOE_ERR_INVALID_ARG, "moe_combine: ksplit = %d outside [1, %d]", ksplit, kMaxKSplit);
    if (!aligned16(y_perm) || !aligned16(out))
        return fail(MOE_ERR_INVALID_ARG, "moe_combine: y_perm and out must be 16-byte aligned");
    int sms;
    if ((rc = check_device(&sms))) return rc;
    return launched(launch_combine(y_perm, w, dest, T, d, top_k, ksplit, static_cast<__nv_bfloat16*>(out), status,
                                   static_cast<cudaStream_t>(stream)),
                    "combine");
}

int moe_forward(const void* x, const float* logits, const void* w_gate_up, const void* w_down, int T, int d,
                int f, int E, int top_k, void* out, void* workspace, size_t workspace_bytes,
                moe_stream_t stream) {
    int rc = check_shape(T, d, f, E, top_k, true);
    if (rc) return rc;
    if (T == 0) return ok();
    if (!x || !logits || !w_gate_up || !w_down || !out)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward: null pointer");
    if (!aligned16(x) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(out))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward: bf16 tensors must be 16-byte aligned");
    const size_t need = layout(T, d, f, E, top_k).total;
    if (!workspace || workspace_bytes < need)
        return fail(MOE_ERR_WORKSPACE, "moe_forward: workspace %zu bytes < %zu needed", workspace_bytes, need);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(MOE_ERR_WORKSPACE, "moe_forward: workspace must be 256-byte aligned");
    int sms;
    if ((rc = check_device(&sms))) return rc;
    return run_layer(x, logits, w_gate_up, w_down, T, d, f, E, top_k, out, workspace, sms,
                     static_cast<cudaStream_t>(stream));
}

int moe_forward_grouped(const void* x, const float* logits, const float* bias, const void* w_gate_up,
                        const void* w_down, int T, int d, int f, int E, int top_k, int n_group, int topk_group,
                        float scale, void* out, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    int rc = check_shape(T, d, f, E, top_k, true);
    if (rc) return rc;
    Router r;
    r.grouped = true;
    r.bias = bias;
    r.n_group = n_group;
    r.topk_group = topk_group;
    r.scale = scale;
    if ((rc = check_router(r, E, top_k, "moe_forward_grouped"))) return rc;
    if (T == 0) return ok();
    if (!x || !logits || !w_gate_up || !w_down || !out)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_grouped: null pointer");
    if (!aligned16(x) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(out))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_grouped: bf16 tensors must be 16-byte aligned");
    const size_t need = layout(T, d, f, E, top_k).total;
    if (!workspace || workspace_bytes < need)
        return fail(MOE_ERR_WORKSPACE, "moe_forward_grouped: workspace %zu bytes < %zu needed", workspace_bytes,
                    need);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(MOE_ERR_WORKSPACE, "moe_forward_grouped: workspace must be 256-byte aligned");
    int sms;
    if ((rc = check_device(&sms))) return rc;
    return run_layer(x, logits, w_gate_up, w_down, T, d, f, E, top_k, out, workspace, sms,
                     static_cast<cudaStream_t>(stream), r);
}

int moe_forward_host(const void* x_host, const float* logits_host, const void* w_gate_up, const void* w_down,
                     int T, int d, int f, int E, int top_k, void* out_host, void* workspace,
                     size_t workspace_bytes, moe_stream_t stream) {
    int rc = check_shape(T, d, f, E, top_k, true);
    if (rc) return rc;
    if (T == 0) return ok();
    if (!x_host || !logits_host || !w_gate_up || !w_down || !out_host)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_host: null pointer");
    const size_t need = layout(T, d, f, E, top_k).total;
    const size_t stage = moe_host_staging_size(T, d, E);
    if (!workspace || workspace_bytes < need + stage)
        return fail(MOE_ERR_WORKSPACE, "moe_forward_host: workspace %zu bytes < %zu needed", workspace_bytes,
                    need + stage);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(MOE_ERR_WORKSPACE, "moe_forward_host: workspace must be 256-byte aligned");
    if (!aligned16(w_gate_up) || !aligned16(w_down))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_host: weights must be 16-byte aligned");
    int sms;
    if ((rc = check_device(&sms))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t xb = static_cast<size_t>(T) * d * 2, lb = static_cast<size_t>(T) * E * 4;
    void* x_dev = at<char>(workspace, need);
    void* out_dev = at<char>(workspace, need + align256(xb));
    float* logits_dev = at<float>(workspace, need + 2 * align256(xb));
    cudaError_t e;
    if ((e = cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(logits_dev, logits_host, lb, cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return fail(MOE_ERR_CUDA, "moe_forward_host: host-to-device copy: %s", cudaGetErrorString(e));
    if ((rc = run_layer(x_dev, logits_dev, w_gate_up, w_down, T, d, f, E, top_k, out_dev, workspace, sms, s)))
        return rc;
    if ((e = cudaMemcpyAsync(out_host, out_dev, xb, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return fail(MOE_ERR_CUDA, "moe_forward_host: device-to-host copy: %s", cudaGetErrorString(e));
    return ok();
}

static int forward_host_batches(const void* const* x_hosts, const float* const* logits_hosts, const void* w_gate_up,
                                const void* w_down, int n_batches, int T, int d, int f, int E, int top_k,
                                void* const* out_hosts, void* workspace, size_t workspace_bytes, moe_stream_t stream,
                                moe_stream_t h2d_stream, moe_stream_t d2h_stream, const Router& router) {
    const char* name = router.grouped ? "moe_forward_grouped_host_batches" : "moe_forward_host_batches";
    int rc = check_shape(T, d, f, E, top_k, true);
    if (rc) return rc;
    if ((rc = check_router(router, E, top_k, name))) return rc;
    if (n_batches < 0) return fail(MOE_ERR_INVALID_ARG, "%s: n_batches = %d < 0", name, n_batches);
    if (T == 0 || n_batches == 0) return ok();
    if ((rc = check_host_batches(name, x_hosts, logits_hosts, out_hosts, n_batches))) return rc;
    if (!w_gate_up || !w_down) return fail(MOE_ERR_INVALID_ARG, "%s: null pointer", name);
    const size_t need = layout(T, d, f, E, top_k).total;
    const size_t stage = moe_host_staging_size(T, d, E);
    if (!workspace || workspace_bytes < need + 2 * stage)
        return fail(MOE_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu needed", name, workspace_bytes, need + 2 * stage);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(MOE_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", name);
    if (!aligned16(w_gate_up) || !aligned16(w_down))
        return fail(MOE_ERR_INVALID_ARG, "%s: weights must be 16-byte aligned", name);
    int sms;
    if ((rc = check_device(&sms))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return run_host_batches(name, x_hosts, logits_hosts, out_hosts, n_batches, T, d, E, need, workspace, s,
                            static_cast<cudaStream_t>(h2d_stream), static_cast<cudaStream_t>(d2h_stream),
                            [&](const void* x, const float* l, void* o) {
                                return run_layer(x, l, w_gate_up, w_down, T, d, f, E, top_k, o, workspace, sms, s,
                                                 router);
                            });
}

int moe_forward_host_batches(const void* const* x_hosts, const float* const* logits_hosts, const void* w_gate_up,
                             const void* w_down, int n_batches, int T, int d, int f, int E, int top_k,
                             void* const* out_hosts, void* workspace, size_t workspace_bytes, moe_stream_t stream,
                             moe_stream_t h2d_stream, moe_stream_t d2h_stream) {
    return forward_host_batches(x_hosts, logits_hosts, w_gate_up, w_down, n_batches, T, d, f, E, top_k, out_hosts,
                                workspace, workspace_bytes, stream, h2d_stream, d2h_stream, Router());
}

int moe_forward_grouped_host_batches(const void* const* x_hosts, const float* const* logits_hosts, const float* bias,
                                     const void* w_gate_up, const void* w_down, int n_batches, int T, int d, int f,
                                     int E, int top_k, int n_group, int topk_group, float scale,
                                     void* const* out_hosts, void* workspace, size_t workspace_bytes,
                                     moe_stream_t stream, moe_stream_t h2d_stream, moe_stream_t d2h_stream) {
    Router r;
    r.grouped = true;
    r.bias = bias;
    r.n_group = n_group;
    r.topk_group = topk_group;
    r.scale = scale;
    return forward_host_batches(x_hosts, logits_hosts, w_gate_up, w_down, n_batches, T, d, f, E, top_k, out_hosts,
                                workspace, workspace_bytes, stream, h2d_stream, d2h_stream, r);
}

int moe_forward_noalloc(const void* x, const float* logits, const void* w_gate_up, const void* w_down, int T,
                        int d, int f, int E, int top_k, void* out, moe_stream_t stream) {
    int rc = check_shape(T, d, f, E, top_k, true);
    if (rc) return rc;
    if (T == 0) return ok();
    if (!x || !logits || !w_gate_up || !w_down || !out)
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_noalloc: null pointer");
    if (!aligned16(x) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(out))
        return fail(MOE_ERR_INVALID_ARG, "moe_forward_noalloc: bf16 tensors must be 16-byte aligned");
    const size_t need = layout(T, d, f, E, top_k).total;
    if (need > MOE_NOALLOC_SCRATCH_BYTES)
        return fail(MOE_ERR_WORKSPACE,
                    "moe_forward_noalloc: this shape needs %zu bytes of scratch, more than the fixed %llu; "
                    "use moe_forward with a workspace",
                    need, static_cast<unsigned long long>(MOE_NOALLOC_SCRATCH_BYTES));
    int sms;
    if ((rc = check_device(&sms))) return rc;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    void* ws = nullptr;
    if ((rc = noalloc_scratch(dev, &ws))) return rc;
    return run_layer(x, logits, w_gate_up, w_down, T, d, f, E, top_k, out, ws, sms,
                     static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------------------------
// FP8 (E4M3) variant
// ---------------------------------------------------------------------------------------------
size_t moe_workspace_size_fp8(int T, int d, int f, int E, int top_k) {
    if (check_shape_fp8(T, d, f, E, top_k, "moe_workspace_size_fp8") != MOE_OK) return 0;
    return layout_fp8(T, d, f, E, top_k).total;
}

int moe_workspace_layout_fp8(int T, int d, int f, int E, int top_k, size_t* offsets_out) {
    int rc = check_shape_fp8(T, d, f, E, top_k, "moe_workspace_layout_fp8");
    if (rc) return rc;
    if (!offsets_out) return fail(MOE_ERR_INVALID_ARG, "moe_workspace_layout_fp8: null pointer");
    const Layout8 L = layout_fp8(T, d, f, E, top_k);
    const size_t v[14] = {L.status, L.idx, L.w, L.counts, L.offsets, L.src, L.dest,
                          L.x8, L.sx, L.h, L.h8, L.sh, L.y_perm, L.total};
    for (int i = 0; i < 14; ++i) offsets_out[i] = v[i];
    return ok();
}

int moe_down_ksplit_fp8(int T, int d, int f, int E, int top_k) {
    if (check_shape_fp8(T, d, f, E, top_k, "moe_down_ksplit_fp8") != MOE_OK) return 0;
    return down_ksplit(T, d, f, E, top_k, true);
}

int moe_gemm_pair_mode_fp8(int T, int d, int f, int E, int top_k, int kind) {
    if (check_shape_fp8(T, d, f, E, top_k, "moe_gemm_pair_mode_fp8") != MOE_OK || (kind != 0 && kind != 1)) return -1;
    return use_pair(static_cast<long long>(T) * top_k, E, kind == 0 ? f : d, kind, true);
}

int moe_forward_fp8_launch_count(int T, int E, int top_k) {
    if (check_shape(T, -1, 0, E, top_k, false) != MOE_OK) return -1;
    if (T == 0) return 0;
    return (fuse_route_permute(T, E) ? 5 : 6) - (fold_combine() ? 1 : 0);
}

int moe_permute_fp8(const int32_t* idx, const void* x, int T, int d, int E, int top_k, int32_t* counts,
                    int32_t* offsets, int32_t* src, int32_t* dest, void* x8_perm, float* sx, int32_t* status,
                    moe_stream_t stream) {
    int rc = check_shape(T, d, 0, E, top_k, false);
    if (rc) return rc;
    if (T == 0) return ok();
    if (!idx || !x || !counts || !offsets || !src || !dest || !x8_perm || !sx)
        return fail(MOE_ERR_INVALID_ARG, "moe_permute_fp8: null pointer");
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(x8_perm) & 7u) || (reinterpret_cast<uintptr_t>(sx) & 3u))
        return fail(MOE_ERR_INVALID_ARG, "moe_permute_fp8: x must be 16-byte, x8_perm 8-byte, sx 4-byte aligned");
    int sms;
    if ((rc = check_device(&sms))) return rc;
    return launched(launch_permute(idx, static_cast<const __nv_bfloat16*>(x), T, d, E, top_k, counts, offsets, src,
                                   dest, nullptr, status, sms, static_cast<cudaStream_t>(stream),
                                   static_cast<uint8_t*>(x8_perm), sx),
                    "permute");
}

int moe_quantize_weights_fp8(const void* W, int E, int K, int N, void* Wq, float* scale, moe_stream_t stream) {
    if (E < 1 || E > kMaxE || !dim_ok(K) || !dim_ok(N) || K % 128 != 0)
        return fail(MOE_ERR_INVALID_ARG,
                    "moe_quantize_weights_fp8: E = %d in [1, %d], K = %d a multiple of 128 and N = %d of 64 "
                    "(both <= %d) required",
                    E, kMaxE, K, N, kMaxDim);
    if (!W || !Wq || !scale) return fail(MOE_ERR_INVALID_ARG, "moe_quantize_weights_fp8: null pointer");
    int sms, rc;
    if ((rc = check_device(&sms))) return rc;
    return launched(launch_quantize_weights_fp8(static_cast<const __nv_bfloat16*>(W), E, K, N,
                                                static_cast<uint8_t*>(Wq), scale, static_cast<cudaStream_t>(stream)),
                    "quantize weights");
}

int moe_quantize_rows_fp8(const void* a, const int32_t* src, int R, int C, int src_rows, void* q, float* scale,
                          int32_t* status, moe_stream_t stream) {
    if (R < 0 || C < 8 || C % 8 != 0 || C > kMaxDim || src_rows < 0 || (!src && src_rows < R))
        return fail(MOE_ERR_INVALID_ARG,
                    "moe_quantize_rows_fp8: R = %d >= 0, C = %d a multiple of 8 in [8, %d], src_rows = %d "
                    "(>= R without src) required",
                    R, C, kMaxDim, src_rows);
    if (R == 0) return ok();
    if (!a || !q || !scale) return fail(MOE_ERR_INVALID_ARG, "moe_quantize_rows_fp8: null pointer");
    if (!aligned16(a) || (reinterpret_cast<uintptr_t>(q) & 7u))
        return fail(MOE_ERR_INVALID_ARG, "moe_quantize_rows_fp8: a must be 16-byte and q 8-byte aligned");
    int sms, rc;
    if ((rc = check_device(&sms))) return rc;
    return launched(launch_quantize_rows_fp8(static_cast<const __nv_bfloat16*>(a), src, R, C, src_rows,
                                             static_cast<uint8_t*>(q), scale, status, static_cast<cudaStream_t>(stream)),
                    "quantize rows");
}

// The FP8 GEMM stage calls; blocks = true for the blockwise kernel.
static int gemm8_entry(int kind, const void* A, const float* sa, const void* B, const float* sb,
                       const int32_t* offsets, int M, int d, int f, int E, int ksplit, void* out, int32_t* status,
                       moe_stream_t stream, const char* name, bool blocks = false, float* h_scale = nullptr) {
    int rc = check_shape_fp8(0, d, f, E, 1, name);
    if (rc) return rc;
    if (M < 0) return fail(MOE_ERR_INVALID_ARG, "%s: M = %d must be >= 0", name, M);
    if (ksplit < 1 || ksplit > kMaxKSplit)
        return fail(MOE_ERR_INVALID_ARG, "%s: ksplit = %d outside [1, %d]", name, ksplit, kMaxKSplit);
    if (M == 0) return ok();
    if (!A || !sa || !B || !sb || !offsets || !out) return fail(MOE_ERR_INVALID_ARG, "%s: null pointer", name);
    if (!aligned16(A) || !aligned16(B) || !aligned16(out))
        return fail(MOE_ERR_INVALID_ARG, "%s: operands must be 16-byte aligned", name);
    if (!aligned16(sb) || (reinterpret_cast<uintptr_t>(sa) & 3u) || (reinterpret_cast<uintptr_t>(h_scale) & 3u))
        return fail(MOE_ERR_INVALID_ARG, "%s: weight scales must be 16-byte, row scales 4-byte aligned", name);
    int sms;
    if ((rc = check_device(&sms))) return rc;
    const int pair = blocks ? 0 : use_pair(M, E, kind == 0 ? f : d, kind, true);
    GemmArgs g = kind == 0 ? GemmArgs{A, B, offsets, M, d, f, E, out, status, 1, swap_max_rows(), pair}
                           : GemmArgs{A, B, offsets, M, f, d, E, out, status, ksplit, swap_max_rows(), pair};
    g.pair_swap_max = pair_swap_max_rows();
    g.pair_layout = pair_layout();
    g.pair_split = pair_split();
    g.fp8 = true;
    g.fp8_blocks = blocks;
    g.a_scale = sa;
    g.b_scale = sb;
    g.h_scale = h_scale;
    const char* why = "";
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = blocks ? launch_grouped_gemm_fp8b(kind, g, sms, cs, &why) : launch_grouped_gemm(kind, g, sms, cs, &why);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s (%s)", name, why, cudaGetErrorString(e));
    return ok();
}

int moe_grouped_gemm_gateup_swiglu_fp8(const void* x8_perm, const float* sx, const void* w8_gate_up,
                                       const float* s_gate_up, const int32_t* offsets, int M, int d, int f, int E,
                                       void* h, int32_t* status, moe_stream_t stream) {
    return gemm8_entry(0, x8_perm, sx, w8_gate_up, s_gate_up, offsets, M, d, f, E, 1, h, status, stream,
                       "moe_grouped_gemm_gateup_swiglu_fp8");
}

int moe_grouped_gemm_down_fp8(const void* h8, const float* sh, const void* w8_down, const float* s_down,
                              const int32_t* offsets, int M, int d, int f, int E, int ksplit, float* y_perm,
                              int32_t* status, moe_stream_t stream) {
    return gemm8_entry(1, h8, sh, w8_down, s_down, offsets, M, d, f, E, ksplit, y_perm, status, stream,
                       "moe_grouped_gemm_down_fp8");
}

// moe_forward_fp8 and moe_forward_fp8b: argument checks, then the layer.
static int forward8_entry(const void* x, const float* logits, const void* w8_gate_up, const float* s_gate_up,
                          const void* w8_down, const float* s_down, int T, int d, int f, int E, int top_k, void* out,
                          void* workspace, size_t workspace_bytes, moe_stream_t stream, bool blocks,
                          const Router& router = Router()) {
    const char* name = router.grouped ? (blocks ? "moe_forward_grouped_fp8b" : "moe_forward_grouped_fp8")
                                      : (blocks ? "moe_forward_fp8b" : "moe_forward_fp8");
    int rc = check_shape_fp8(T, d, f, E, top_k, name);
    if (rc) return rc;
    if ((rc = check_router(router, E, top_k, name))) return rc;
    if (T == 0) return ok();
    if (!x || !logits || !w8_gate_up || !s_gate_up || !w8_down || !s_down || !out)
        return fail(MOE_ERR_INVALID_ARG, "%s: null pointer", name);
    if (!aligned16(x) || !aligned16(w8_gate_up) || !aligned16(w8_down) || !aligned16(out) || !aligned16(s_gate_up) ||
        !aligned16(s_down))
        return fail(MOE_ERR_INVALID_ARG, "%s: tensors and weight scales must be 16-byte aligned", name);
    const size_t need = layout_fp8(T, d, f, E, top_k, blocks).total;
    if (!workspace || workspace_bytes < need)
        return fail(MOE_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu needed", name, workspace_bytes, need);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(MOE_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", name);
    int sms;
    if ((rc = check_device(&sms))) return rc;
    return run_layer_fp8(x, logits, w8_gate_up, s_gate_up, w8_down, s_down, T, d, f, E, top_k, out, workspace, sms,
                         static_cast<cudaStream_t>(stream), blocks, router);
}

// The FP8 layers over host batches (moe_forward_host_batches with moe_forward_fp8[b] as the layer).
static int forward8_host_batches(const void* const* x_hosts, const float* const* logits_hosts, const void* w8_gate_up,
                                 const float* s_gate_up, const void* w8_down, const float* s_down, int n_batches, int T,
                                 int d, int f, int E, int top_k, void* const* out_hosts, void* workspace,
                                 size_t workspace_bytes, moe_stream_t stream, moe_stream_t h2d_stream,
                                 moe_stream_t d2h_stream, bool blocks, const Router& router = Router()) {
    const char* name = router.grouped ? (blocks ? "moe_forward_grouped_fp8b_host_batches"
                                                : "moe_forward_grouped_fp8_host_batches")
                                      : (blocks ? "moe_forward_fp8b_host_batches" : "moe_forward_fp8_host_batches");
    int rc = check_shape_fp8(T, d, f, E, top_k, name);
    if (rc) return rc;
    if ((rc = check_router(router, E, top_k, name))) return rc;
    if (n_batches < 0) return fail(MOE_ERR_INVALID_ARG, "%s: n_batches = %d < 0", name, n_batches);
    if (T == 0 || n_batches == 0) return ok();
    if ((rc = check_host_batches(name, x_hosts, logits_hosts, out_hosts, n_batches))) return rc;
    if (!w8_gate_up || !s_gate_up || !w8_down || !s_down) return fail(MOE_ERR_INVALID_ARG, "%s: null pointer", name);
    if (!aligned16(w8_gate_up) || !aligned16(w8_down) || !aligned16(s_gate_up) || !aligned16(s_down))
        return fail(MOE_ERR_INVALID_ARG, "%s: weights and weight scales must be 16-byte aligned", name);
    const size_t need = layout_fp8(T, d, f, E, top_k, blocks).total;
    const size_t stage = moe_host_staging_size(T, d, E);
    if (!workspace || workspace_bytes < need + 2 * stage)
        return fail(MOE_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu needed", name, workspace_bytes, need + 2 * stage);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(MOE_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", name);
    int sms;
    if ((rc = check_device(&sms))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return run_host_batches(name, x_hosts, logits_hosts, out_hosts, n_batches, T, d, E, need, workspace, s,
                            static_cast<cudaStream_t>(h2d_stream), static_cast<cudaStream_t>(d2h_stream),
                            [&](const void* x, const float* l, void* o) {
                                return run_layer_fp8(x, l, w8_gate_up, s_gate_up, w8_down, s_down, T, d, f, E, top_k,
                                                     o, workspace, sms, s, blocks, router);
                            });
}

int moe_forward_fp8_host_batches(const void* const* x_hosts, const float* const* logits_hosts, const void* w8_gate_up,
                                 const float* s_gate_up, const void* w8_down, const float* s_down, int n_batches, int T,
                                 int d, int f, int E, int top_k, void* const* out_hosts, void* workspace,
                                 size_t workspace_bytes, moe_stream_t stream, moe_stream_t h2d_stream,
                                 moe_stream_t d2h_stream) {
    return forward8_host_batches(x_hosts, logits_hosts, w8_gate_up, s_gate_up, w8_down, s_down, n_batches, T, d, f, E,
                                 top_k, out_hosts, workspace, workspace_bytes, stream, h2d_stream, d2h_stream, false);
}

int moe_forward_fp8b_host_batches(const void* const* x_hosts, const float* const* logits_hosts,
                                  const void* w8_gate_up, const float* s_gate_up, const void* w8_down,
                                  const float* s_down, int n_batches, int T, int d, int f, int E, int top_k,
                                  void* const* out_hosts, void* workspace, size_t workspace_bytes, moe_stream_t stream,
                                  moe_stream_t h2d_stream, moe_stream_t d2h_stream) {
    return forward8_host_batches(x_hosts, logits_hosts, w8_gate_up, s_gate_up, w8_down, s_down, n_batches, T, d, f, E,
                                 top_k, out_hosts, workspace, workspace_bytes, stream, h2d_stream, d2h_stream, true);
}

static Router grouped_router(const float* bias, int n_group, int topk_group, float scale) {
    Router r;
    r.grouped = true;
    r.bias = bias;
    r.n_group = n_group;
    r.topk_group = topk_group;
    r.scale = scale;
    return r;
}

int moe_forward_grouped_fp8_host_batches(const void* const* x_hosts, const float* const* logits_hosts,
                                         const float* bias, const void* w8_gate_up, const float* s_gate_up,
                                         const void* w8_down, const float* s_down, int n_batches, int T, int d, int f,
                                         int E, int top_k, int n_group, int topk_group, float scale,
                                         void* const* out_hosts, void* workspace, size_t workspace_bytes,
                                         moe_stream_t stream, moe_stream_t h2d_stream, moe_stream_t d2h_stream) {
    return forward8_host_batches(x_hosts, logits_hosts, w8_gate_up, s_gate_up, w8_down, s_down, n_batches, T, d, f, E,
                                 top_k, out_hosts, workspace, workspace_bytes, stream, h2d_stream, d2h_stream, false,
                                 grouped_router(bias, n_group, topk_group, scale));
}

int moe_forward_grouped_fp8b_host_batches(const void* const* x_hosts, const float* const* logits_hosts,
                                          const float* bias, const void* w8_gate_up, const float* s_gate_up,
                                          const void* w8_down, const float* s_down, int n_batches, int T, int d,
                                          int f, int E, int top_k, int n_group, int topk_group, float scale,
                                          void* const* out_hosts, void* workspace, size_t workspace_bytes,
                                          moe_stream_t stream, moe_stream_t h2d_stream, moe_stream_t d2h_stream) {
    return forward8_host_batches(x_hosts, logits_hosts, w8_gate_up, s_gate_up, w8_down, s_down, n_batches, T, d, f, E,
                                 top_k, out_hosts, workspace, workspace_bytes, stream, h2d_stream, d2h_stream, true,
                                 grouped_router(bias, n_group, topk_group, scale));
}

int moe_forward_grouped_fp8(const void* x, const float* logits, const float* bias, const void* w8_gate_up,
                            const float* s_gate_up, const void* w8_down, const float* s_down, int T, int d, int f,
                            int E, int top_k, int n_group, int topk_group, float scale, void* out, void* workspace,
                            size_t workspace_bytes, moe_stream_t stream) {
    return forward8_entry(x, logits, w8_gate_up, s_gate_up, w8_down, s_down, T, d, f, E, top_k, out, workspace,
                          workspace_bytes, stream, false, grouped_router(bias, n_group, topk_group, scale));
}

int moe_forward_grouped_fp8b(const void* x, const float* logits, const float* bias, const void* w8_gate_up,
                             const float* s_gate_up, const void* w8_down, const float* s_down, int T, int d, int f,
                             int E, int top_k, int n_group, int topk_group, float scale, void* out, void* workspace,
                             size_t workspace_bytes, moe_stream_t stream) {
    return forward8_entry(x, logits, w8_gate_up, s_gate_up, w8_down, s_down, T, d, f, E, top_k, out, workspace,
                          workspace_bytes, stream, true, grouped_router(bias, n_group, topk_group, scale));
}

int moe_forward_fp8(const void* x, const float* logits, const void* w8_gate_up, const float* s_gate_up,
                    const void* w8_down, const float* s_down, int T, int d, int f, int E, int top_k, void* out,
                    void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    return forward8_entry(x, logits, w8_gate_up, s_gate_up, w8_down, s_down, T, d, f, E, top_k, out, workspace,
                          workspace_bytes, stream, false);
}

// ---------------------------------------------------------------------------------------------
// Blockwise FP8 variant (1 x 128 activation blocks, 128 x 128 weight blocks, power-of-two scales)
// ---------------------------------------------------------------------------------------------
size_t moe_workspace_size_fp8b(int T, int d, int f, int E, int top_k) {
    if (check_shape_fp8(T, d, f, E, top_k, "moe_workspace_size_fp8b") != MOE_OK) return 0;
    return layout_fp8(T, d, f, E, top_k, true).total;
}

int moe_workspace_layout_fp8b(int T, int d, int f, int E, int top_k, size_t* offsets_out) {
    int rc = check_shape_fp8(T, d, f, E, top_k, "moe_workspace_layout_fp8b");
    if (rc) return rc;
    if (!offsets_out) return fail(MOE_ERR_INVALID_ARG, "moe_workspace_layout_fp8b: null pointer");
    const Layout8 L = layout_fp8(T, d, f, E, top_k, true);
    const size_t v[14] = {L.status, L.idx, L.w, L.counts, L.offsets, L.src, L.dest,
                          L.x8, L.sx, L.h, L.h8, L.sh, L.y_perm, L.total};
    for (int i = 0; i < 14; ++i) offsets_out[i] = v[i];
    return ok();
}

int moe_down_ksplit_fp8b(int T, int d, int f, int E, int top_k) {
    if (check_shape_fp8(T, d, f, E, top_k, "moe_down_ksplit_fp8b") != MOE_OK) return 0;
    return down_ksplit(T, d, f, E, top_k, true, true);
}

int moe_forward_fp8b_launch_count(int T, int E, int top_k) {
    if (check_shape(T, -1, 0, E, top_k, false) != MOE_OK) return -1;
    if (T == 0) return 0;
    return (fuse_route_permute(T, E) ? 5 : 6) + (fp8b_fuse_h(static_cast<long long>(T) * top_k, E) ? 0 : 1);
}

int moe_fp8b_gemm_quantizes_h(int T, int E, int top_k) {
    if (check_shape(T, -1, 0, E, top_k, false) != MOE_OK) return -1;
    return fp8b_fuse_h(static_cast<long long>(T) * top_k, E) ? 1 : 0;
}

int moe_quantize_weights_fp8b(const void* W, int E, int K, int N, void* Wq, float* scale, moe_stream_t stream) {
    if (E < 1 || E > kMaxE || !dim_ok(K) || !dim_ok(N) || K % 128 != 0 || N % 128 != 0)
        return fail(MOE_ERR_INVALID_ARG,
                    "moe_quantize_weights_fp8b: E = %d in [1, %d], K = %d and N = %d multiples of 128 "
                    "(<= %d) required",
                    E, kMaxE, K, N, kMaxDim);
    if (!W || !Wq || !scale) return fail(MOE_ERR_INVALID_ARG, "moe_quantize_weights_fp8b: null pointer");
    if (!aligned16(W) || !aligned16(Wq) || (reinterpret_cast<uintptr_t>(scale) & 3u))
        return fail(MOE_ERR_INVALID_ARG, "moe_quantize_weights_fp8b: W and Wq 16-byte, scale 4-byte aligned");
    int sms, rc;
    if ((rc = check_device(&sms))) return rc;
    return launched(launch_quantize_weights_fp8b(static_cast<const __nv_bfloat16*>(W), E, K, N,
                                                 static_cast<uint8_t*>(Wq), scale, static_cast<cudaStream_t>(stream)),
                    "quantize weights (blockwise)");
}

int moe_quantize_rows_fp8b(const void* a, const int32_t* src, int R, int C, int src_rows, void* q, float* scale,
                           int32_t* status, moe_stream_t stream) {
    if (R < 0 || C < 128 || C % 128 != 0 || C > kMaxDim || src_rows < 0 || (!src && src_rows < R))
        return fail(MOE_ERR_INVALID_ARG,
                    "moe_quantize_rows_fp8b: R = %d >= 0, C = %d a multiple of 128 in [128, %d], src_rows = %d "
                    "(>= R without src) required",
                    R, C, kMaxDim, src_rows);
    if (R == 0) return ok();
    if (!a || !q || !scale) return fail(MOE_ERR_INVALID_ARG, "moe_quantize_rows_fp8b: null pointer");
    if (!aligned16(a) || (reinterpret_cast<uintptr_t>(q) & 7u) || (reinterpret_cast<uintptr_t>(scale) & 3u))
        return fail(MOE_ERR_INVALID_ARG, "moe_quantize_rows_fp8b: a 16-byte, q 8-byte, scale 4-byte aligned");
    int sms, rc;
    if ((rc = check_device(&sms))) return rc;
    return launched(launch_quantize_rows_fp8b(static_cast<const __nv_bfloat16*>(a), src, R, C, src_rows,
                                              static_cast<uint8_t*>(q), scale, status,
                                              static_cast<cudaStream_t>(stream)),
                    "quantize rows (blockwise)");
}

int moe_grouped_gemm_gateup_swiglu_fp8b(const void* x8_perm, const float* sx, const void* w8_gate_up,
                                        const float* s_gate_up, const int32_t* offsets, int M, int d, int f, int E,
                                        void* h, int32_t* status, moe_stream_t stream) {
    return gemm8_entry(0, x8_perm, sx, w8_gate_up, s_gate_up, offsets, M, d, f, E, 1, h, status, stream,
                       "moe_grouped_gemm_gateup_swiglu_fp8b", true);
}

int moe_grouped_gemm_gateup_swiglu_fp8b_q(const void* x8_perm, const float* sx, const void* w8_gate_up,
                                          const float* s_gate_up, const int32_t* offsets, int M, int d, int f, int E,
                                          void* h8, float* sh, int32_t* status, moe_stream_t stream) {
    const char* name = "moe_grouped_gemm_gateup_swiglu_fp8b_q";
    if (M > 0 && !sh) return fail(MOE_ERR_INVALID_ARG, "%s: null pointer", name);
    return gemm8_entry(0, x8_perm, sx, w8_gate_up, s_gate_up, offsets, M, d, f, E, 1, h8, status, stream, name, true,
                       sh);
}

int moe_grouped_gemm_down_fp8b(const void* h8, const float* sh, const void* w8_down, const float* s_down,
                               const int32_t* offsets, int M, int d, int f, int E, int ksplit, float* y_perm,
                               int32_t* status, moe_stream_t stream) {
    return gemm8_entry(1, h8, sh, w8_down, s_down, offsets, M, d, f, E, ksplit, y_perm, status, stream,
                       "moe_grouped_gemm_down_fp8b", true);
}

int moe_forward_fp8b(const void* x, const float* logits, const void* w8_gate_up, const float* s_gate_up,
                     const void* w8_down, const float* s_down, int T, int d, int f, int E, int top_k, void* out,
                     void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    return forward8_entry(x, logits, w8_gate_up, s_gate_up, w8_down, s_down, T, d, f, E, top_k, out, workspace,
                          workspace_bytes, stream, true);
}

int moe_get_device_error(const void* status_or_workspace, int32_t* code) {
    if (!code) return fail(MOE_ERR_INVALID_ARG, "moe_get_device_error: null pointer");
    if (!status_or_workspace) {  // the status word of moe_forward_noalloc's array on the current device
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "moe_get_device_error: %s", cudaGetErrorString(e));
        void* ws = nullptr;
        int rc = noalloc_scratch(dev, &ws);
        if (rc) return rc;
        status_or_workspace = static_cast<const unsigned char*>(ws) + layout(1, 64, 64, 1, 1).status;
    }
    cudaError_t e = cudaMemcpy(code, status_or_workspace, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "moe_get_device_error: %s", cudaGetErrorString(e));
    return ok();
}

}  // extern "C"
