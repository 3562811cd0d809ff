// permute.cu — step 2: group the T*k (token, slot) assignments by expert and copy x rows into
// that order (the "dispatch" / data rearrangement ahead of the grouped GEMM: DeepGEMM PR #304
// write-up, section 3.1, m-grouped contiguous layout; HPC-Ops page, FusedMoE paragraph).
//
// Order: expert ascending, then token ascending — a stable counting sort, so every output is
// unique and the kernel is bit-exact with any correct implementation.
//
// One launch, no grid-wide synchronisation: every block histograms ALL assignments itself (a
// few tens of KB of idx, read from L2), which gives it both the global offsets and, for its own
// chunk of tokens, how many earlier tokens chose each expert.  It then ranks its chunk's
// assignments, writes src/dest, and copies its tokens' x rows to their k destinations with
// 16-byte vector loads and stores.
#include <cstdlib>

#include "common.cuh"
#include "fp8.cuh"

namespace moe {
namespace {

constexpr int kMaxE = 256;
constexpr int kMaxK = 8;
constexpr int kMaxTokPerBlock = 64;
constexpr int kCopyBatch = 4;
constexpr long long kFuseMaxLogits = 8192;  // route+permute fusion: T*E at most this

// FP8 layer: instead of copying x rows, quantise each of the chunk's tokens once (absmax over its d
// values, fp8.cuh's per-row arithmetic) and write its codes and scale to each of its k permuted
// rows (rows < 0, from an invalid expert id, are skipped).  The block splits into 1, 2, 4 or 8
// teams, one token per team at a time, so a block with a single token still spreads its row over
// all the block's threads: a pass for the absmax (team reduction through shared memory), a second (from
// L1) for the codes.  Called by every thread of the block.
template <int kPermThreads>
__device__ __forceinline__ void quantize_perm_rows(const uint4* __restrict__ x, int t0, int t1, int d, int k,
                                                   const int* crow, uint2* __restrict__ x8, float* __restrict__ sx,
                                                   float* red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ntok = t1 - t0, dv = d / 8;
    int teams = 1;
    while (teams < ntok && teams < kPermThreads / 32) teams <<= 1;
    const int team_threads = kPermThreads / teams, team = tid / team_threads, tt = tid % team_threads;
    const int wpt = team_threads / 32;  // warps per team
    for (int base = 0; base < ntok; base += teams) {  // uniform trip count: every thread reaches the barriers
        const int tl = base + team;
        const uint4* row = x + static_cast<size_t>(t0 + (tl < ntok ? tl : 0)) * dv;
        float m = 0.0f;
        if (tl < ntok)
            for (int v = tt; v < dv; v += team_threads) m = fmaxf(m, absmax8(__ldg(row + v)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) red[warp] = m;
        __syncthreads();
        m = 0.0f;
        for (int i = 0; i < wpt; ++i) m = fmaxf(m, red[team * wpt + i]);
        if (tl < ntok) {
            const float inv = fp8_inv(m);
            if (tt < k) {
                const int r = crow[tl * k + tt];
                if (r >= 0) sx[r] = fp8_scale(m);
            }
            for (int v = tt; v < dv; v += team_threads) {
                const uint2 c = codes8(__ldg(row + v), inv);
                for (int j = 0; j < k; ++j) {
                    const int r = crow[tl * k + j];
                    if (r >= 0) x8[static_cast<size_t>(r) * dv + v] = c;
                }
            }
        }
        __syncthreads();  // red is rewritten next round
    }
}

template <int kPermThreads>
__global__ void __launch_bounds__(kPermThreads)
permute_kernel(const int32_t* __restrict__ idx, const uint4* __restrict__ x, int T, int d, int E,
               int k, int tok_per_block, int32_t* __restrict__ counts,
               int32_t* __restrict__ offsets, int32_t* __restrict__ src,
               int32_t* __restrict__ dest, uint4* __restrict__ x_perm, uint2* __restrict__ x8,
               float* __restrict__ sx, int32_t* __restrict__ status, int32_t* __restrict__ fold_cnt,
               int fold_nblk) {
    __shared__ int tot[kMaxE];      // assignments per expert, all tokens
    __shared__ int before[kMaxE];   // ... from tokens before this block's chunk
    __shared__ int off[kMaxE + 1];  // exclusive scan of tot
    __shared__ int cidx[kMaxTokPerBlock * kMaxK];
    __shared__ int crow[kMaxTokPerBlock * kMaxK];
    __shared__ int bad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_trigger();
    for (int e = tid; e < E; e += kPermThreads) {
        tot[e] = 0;
        before[e] = 0;
    }
    if (tid == 0) bad = 0;
    __syncthreads();

    const int t0 = blockIdx.x * tok_per_block;
    const int t1 = min(T, t0 + tok_per_block);
    const int nA = T * k, a0 = t0 * k;
    // The down GEMM's combine-fold counters of this block's tokens start at zero.
    if (fold_cnt != nullptr)
        for (int i = tid; i < (t1 - t0) * fold_nblk; i += kPermThreads)
            fold_cnt[static_cast<size_t>(t0) * fold_nblk + i] = 0;

    // Histogram of all assignments (tot) and of those before this block's chunk (before).
    if (E <= 32) {
        // Few experts: lanes collide often, so aggregate equal ids within the warp first.  The
        // trip count is warp-uniform so __match_any_sync sees all 32 lanes.
        for (int base = warp * 32; base < nA; base += kPermThreads) {
            const int a = base + lane;
            const int e = a < nA ? __ldg(idx + a) : 0;
            const bool ok = a < nA && static_cast<unsigned>(e) < static_cast<unsigned>(E);
            if (a < nA && !ok) bad = 1;
            const int key = ok ? (e * 2 + (a < a0 ? 1 : 0)) : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, key);
            if (ok && lane == __ffs(peers) - 1) {
                atomicAdd(&tot[e], __popc(peers));
                if (a < a0) atomicAdd(&before[e], __popc(peers));
            }
        }
    } else {
        // Many experts: collisions are rare; 16-byte loads of four ids, plain shared atomics.
        const bool vec = (reinterpret_cast<uintptr_t>(idx) & 15u) == 0;
        const int n4 = vec ? nA / 4 : 0;
        for (int q = tid; q < n4; q += kPermThreads) {
            const int4 v = __ldg(reinterpret_cast<const int4*>(idx) + q);
            const int ev[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = 4 * q + u, e = ev[u];
                if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
                    atomicAdd(&tot[e], 1);
                    if (a < a0) atomicAdd(&before[e], 1);
                } else {
                    bad = 1;
                }
            }
        }
        for (int a = 4 * n4 + tid; a < nA; a += kPermThreads) {
            const int e = __ldg(idx + a);
            if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
                atomicAdd(&tot[e], 1);
                if (a < a0) atomicAdd(&before[e], 1);
            } else {
                bad = 1;
            }
        }
    }
    __syncthreads();

    // Exclusive scan of tot over E <= 256 experts by warp 0, 8 experts per lane.
    if (warp == 0) {
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int sum = 0;
        for (int e = e0; e < e1; ++e) sum += tot[e];
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        int run = incl - sum;
        for (int e = e0; e < e1; ++e) {
            off[e] = run;
            run += tot[e];
        }
        if (lane == 31) off[E] = incl;
    }
    __syncthreads();

    if (blockIdx.x == 0) {
        for (int e = tid; e < E; e += kPermThreads) counts[e] = tot[e];
        for (int e = tid; e <= E; e += kPermThreads) offsets[e] = off[e];
    }

    // Rank this chunk's assignments.  Each expert occurs at most once per token, so the rank of
    // (t, j) within expert e = number of earlier chunk tokens that chose e.
    const int nloc = (t1 - t0) * k;
    if (tid < nloc) cidx[tid] = __ldg(idx + a0 + tid);
    __syncthreads();
    if (tid < nloc) {
        const int e = cidx[tid];
        const int tl = tid / k;
        int row = -1;
        if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
            int rank = 0;
            for (int i = 0; i < tl * k; ++i) rank += (cidx[i] == e);
            for (int i = tl * k; i < tl * k + k; ++i)
                if (i != tid && cidx[i] == e) bad = 1;  // repeated within one token
            row = off[e] + before[e] + rank;
            src[row] = t0 + tl;
        }
        dest[a0 + tid] = row;
        crow[tid] = row;
    }
    __syncthreads();
    if (bad && tid == 0) flag_status(status, MOE_STATUS_BAD_EXPERT_ID);

    if (x8 != nullptr) {
        __shared__ float red[kPermThreads / 32];
        quantize_perm_rows<kPermThreads>(x, t0, t1, d, k, crow, x8, sx, red);
        return;
    }
    // Row copies: x[t] -> x_perm[row(t, j)] for each slot j, 16 bytes per access.  Each thread
    // first issues kCopyBatch independent loads, then their k stores each, so that enough reads
    // are in flight to cover the memory latency.
    if (x_perm == nullptr) return;  // the gate+up GEMM gathers x rows itself
    const int dv = d / 8;  // uint4 per row
    const int nvec = (t1 - t0) * dv;
    for (int base = tid; base < nvec; base += kPermThreads * kCopyBatch) {
        uint4 val[kCopyBatch];
#pragma unroll
        for (int u = 0; u < kCopyBatch; ++u) {
            const int i = base + u * kPermThreads;
            if (i < nvec) {
                const int tl = i / dv, v = i - tl * dv;
                val[u] = __ldg(x + static_cast<size_t>(t0 + tl) * dv + v);
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyBatch; ++u) {
            const int i = base + u * kPermThreads;
            if (i < nvec) {
                const int tl = i / dv, v = i - tl * dv;
                for (int j = 0; j < k; ++j) {
                    const int r = crow[tl * k + j];
                    if (r >= 0) x_perm[static_cast<size_t>(r) * dv + v] = val[u];
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Steps 1 and 2 in one launch, for small routing problems (E <= 32, T*E <= kFuseMaxLogits).
// Every block routes ALL T tokens itself — a thread per token, the softmax router's selection
// (k largest logits, equal logits -> lower id, slot order descending) — to build the histogram
// the permutation needs, so no grid-wide synchronisation is required; it writes idx and w only
// for its own chunk of tokens, then ranks and copies that chunk exactly as permute_kernel does.
// The redundant routing reads T*E*4 bytes per block from L2 (at most 32 KB).  Measured on the
// Mixtral shape (ms/layer, fused vs two launches): T=32 0.409 vs 0.413, T=512 0.512 vs 0.516,
// T=4096 2.007 vs 1.992 — hence the limit T*E <= 8192.
// ---------------------------------------------------------------------------------------------
constexpr int kFuseMaxE = 32;

__device__ __forceinline__ bool logit_before(float av, int ai, float bv, int bi) {
    const bool an = av != av, bn = bv != bv;  // a NaN ranks below every number, NaNs by id
    if (an != bn) return bn;
    return av > bv || ((av == bv || an) && ai < bi);
}

template <int kPermThreads>
__global__ void __launch_bounds__(kPermThreads)
route_permute_kernel(const float* __restrict__ logits, const uint4* __restrict__ x, int T, int d, int E, int k,
                     int tok_per_block, int32_t* __restrict__ idx, float* __restrict__ w,
                     int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ src,
                     int32_t* __restrict__ dest, uint4* __restrict__ x_perm, uint2* __restrict__ x8,
                     float* __restrict__ sx, int32_t* __restrict__ status, int32_t* __restrict__ fold_cnt,
                     int fold_nblk) {
    __shared__ int tot[kFuseMaxE];
    __shared__ int before[kFuseMaxE];
    __shared__ int off[kFuseMaxE + 1];
    __shared__ int cidx[kMaxTokPerBlock * kMaxK];
    __shared__ int crow[kMaxTokPerBlock * kMaxK];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_trigger();
    if (status != nullptr && blockIdx.x == 0 && tid == 0) *status = 0;  // first kernel of the layer
    if (tid < E) {
        tot[tid] = 0;
        before[tid] = 0;
    }
    __syncthreads();
    const int t0 = blockIdx.x * tok_per_block;
    const int t1 = min(T, t0 + tok_per_block);
    if (fold_cnt != nullptr)  // the down GEMM's combine-fold counters of this block's tokens
        for (int i = tid; i < (t1 - t0) * fold_nblk; i += kPermThreads)
            fold_cnt[static_cast<size_t>(t0) * fold_nblk + i] = 0;

    // Route every token (thread per token); warp-aggregated histogram updates.
    for (int base = warp * 32; base < T; base += kPermThreads) {
        const int t = base + lane;
        const bool active = t < T;
        int sel[kMaxK];
        float selv[kMaxK];
        unsigned used = 0u;
        const float* row = logits + static_cast<size_t>(active ? t : 0) * E;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            sel[j] = 0;
            selv[j] = 0.0f;
            if (j < k) {
                int bi = -1;
                float bv = 0.0f;
                for (int e = 0; e < E; ++e) {
                    const float v = __ldg(row + e);
                    if (!(used & (1u << e)) && (bi < 0 || logit_before(v, e, bv, bi))) {
                        bi = e;
                        bv = v;
                    }
                }
                used |= 1u << bi;
                sel[j] = bi;
                selv[j] = bv;
            }
        }
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j < k) {
                const int key = active ? (sel[j] * 2 + (t < t0 ? 1 : 0)) : -1;
                const unsigned peers = __match_any_sync(0xffffffffu, key);
                if (active && lane == __ffs(peers) - 1) {
                    atomicAdd(&tot[sel[j]], __popc(peers));
                    if (t < t0) atomicAdd(&before[sel[j]], __popc(peers));
                }
            }
        }
        if (active && t >= t0 && t < t1) {
            // Weights of the block's own tokens: softmax restricted to the chosen k.
            float ex[kMaxK], sum = 0.0f;
#pragma unroll
            for (int j = 0; j < kMaxK; ++j) {
                ex[j] = 0.0f;
                if (j < k) {
                    ex[j] = expf(selv[j] - selv[0]);
                    sum += ex[j];
                }
            }
#pragma unroll
            for (int j = 0; j < kMaxK; ++j)
                if (j < k) {
                    idx[static_cast<size_t>(t) * k + j] = sel[j];
                    w[static_cast<size_t>(t) * k + j] = ex[j] / sum;
                    cidx[(t - t0) * k + j] = sel[j];
                }
        }
    }
    __syncthreads();

    // Exclusive scan of tot (E <= 32: one expert per lane of warp 0).
    if (warp == 0) {
        const int v = lane < E ? tot[lane] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane < E) off[lane] = incl - v;
        if (lane == 31) off[E] = incl;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        if (tid < E) counts[tid] = tot[tid];
        if (tid <= E) offsets[tid] = off[tid];
    }

    // Rank this chunk's assignments (ids are valid by construction) and copy its rows.
    const int nloc = (t1 - t0) * k, a0 = t0 * k;
    if (tid < nloc) {
        const int e = cidx[tid];
        const int tl = tid / k;
        int rank = 0;
        for (int i = 0; i < tl * k; ++i) rank += (cidx[i] == e);
        const int row = off[e] + before[e] + rank;
        src[row] = t0 + tl;
        dest[a0 + tid] = row;
        crow[tid] = row;
    }
    __syncthreads();
    if (x8 != nullptr) {
        __shared__ float red[kPermThreads / 32];
        quantize_perm_rows<kPermThreads>(x, t0, t1, d, k, crow, x8, sx, red);
        return;
    }
    if (x_perm == nullptr) return;  // the gate+up GEMM gathers x rows itself
    const int dv = d / 8;
    const int nvec = (t1 - t0) * dv;
    for (int base = tid; base < nvec; base += kPermThreads * kCopyBatch) {
        uint4 val[kCopyBatch];
#pragma unroll
        for (int u = 0; u < kCopyBatch; ++u) {
            const int i = base + u * kPermThreads;
            if (i < nvec) {
                const int tl = i / dv, v = i - tl * dv;
                val[u] = __ldg(x + static_cast<size_t>(t0 + tl) * dv + v);
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyBatch; ++u) {
            const int i = base + u * kPermThreads;
            if (i < nvec) {
                const int tl = i / dv, v = i - tl * dv;
                for (int j = 0; j < k; ++j) x_perm[static_cast<size_t>(crow[tl * k + j]) * dv + v] = val[u];
            }
        }
    }
}

}  // namespace

bool route_permute_fusable(int T, int E) {
    return E <= kFuseMaxE && static_cast<long long>(T) * E <= kFuseMaxLogits;
}

// Threads per permutation block.  Every block histograms all T*k assignments itself, so fewer,
// larger blocks repeat that work fewer times: with E <= 32 (the warp-aggregated histogram) the
// kernel uses 1024-thread blocks, one per SM, else 256-thread blocks, four per SM.  Measured
// (ms/layer, 256 -> 1024 threads): Mixtral shape T=4096 1.938 -> 1.925 (permute 37 -> 27 us), e4m3
// 1.127 -> 1.116, T=512 and T=32 unchanged; softmax-routed DeepSeek shape (E=256) 2.102 -> 2.155
// although its permute alone ran 59 -> 53 us, DeepSeek-V3 router 1.574 -> 1.570.
// MOE_PERM_THREADS=256/512/1024 overrides the choice.
static int perm_threads(int E) {
    const char* v = std::getenv("MOE_PERM_THREADS");
    const int n = v ? std::atoi(v) : 0;
    if (n == 256 || n == 512 || n == 1024) return n;
    return E <= 32 ? 1024 : 256;
}

// Tokens per block: the grid fills the GPU with 256-thread blocks four to an SM (or the same threads
// as fewer, larger blocks), at most kMaxTokPerBlock tokens and at most one assignment per thread.
static int perm_tokens_per_block(int T, int num_sms, int nt) {
    const int per_sm = 1024 / nt;
    const int cap = nt == 256 ? 16 : kMaxTokPerBlock;
    int tpb = (T + per_sm * num_sms - 1) / (per_sm * num_sms);
    return tpb < 1 ? 1 : (tpb > cap ? cap : tpb);
}

template <int NT>
static cudaError_t launch_route_permute_nt(const float* logits, const __nv_bfloat16* x, int T, int d, int E, int k,
                                           int32_t* idx, float* w, int32_t* counts, int32_t* offsets, int32_t* src,
                                           int32_t* dest, __nv_bfloat16* x_perm, int32_t* status, int num_sms,
                                           cudaStream_t s, uint8_t* x8, float* sx, int32_t* fold_cnt, int fold_nblk) {
    const int tpb = perm_tokens_per_block(T, num_sms, NT);
    const int blocks = (T + tpb - 1) / tpb;
    return launch_k(kPdlRoute, route_permute_kernel<NT>, dim3(blocks), dim3(NT), 0, s, logits,
                    reinterpret_cast<const uint4*>(x), T, d, E, k, tpb, idx, w, counts, offsets, src, dest,
                    reinterpret_cast<uint4*>(x_perm), reinterpret_cast<uint2*>(x8), sx, status, fold_cnt, fold_nblk);
}

cudaError_t launch_route_permute(const float* logits, const __nv_bfloat16* x, int T, int d, int E, int k,
                                 int32_t* idx, float* w, int32_t* counts, int32_t* offsets, int32_t* src,
                                 int32_t* dest, __nv_bfloat16* x_perm, int32_t* status, int num_sms,
                                 cudaStream_t s, uint8_t* x8, float* sx, int32_t* fold_cnt, int fold_nblk) {
    switch (perm_threads(E)) {
        case 1024:
            return launch_route_permute_nt<1024>(logits, x, T, d, E, k, idx, w, counts, offsets, src, dest, x_perm,
                                                 status, num_sms, s, x8, sx, fold_cnt, fold_nblk);
        case 512:
            return launch_route_permute_nt<512>(logits, x, T, d, E, k, idx, w, counts, offsets, src, dest, x_perm,
                                                status, num_sms, s, x8, sx, fold_cnt, fold_nblk);
        default:
            return launch_route_permute_nt<256>(logits, x, T, d, E, k, idx, w, counts, offsets, src, dest, x_perm,
                                                status, num_sms, s, x8, sx, fold_cnt, fold_nblk);
    }
}

template <int NT>
static cudaError_t launch_permute_nt(const int32_t* idx, const __nv_bfloat16* x, int T, int d, int E, int k,
                                     int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dest,
                                     __nv_bfloat16* x_perm, int32_t* status, int num_sms, cudaStream_t s, uint8_t* x8,
                                     float* sx, int32_t* fold_cnt, int fold_nblk) {
    const int tpb = perm_tokens_per_block(T, num_sms, NT);
    const int blocks = (T + tpb - 1) / tpb;
    return launch_k(kPdlPermute, permute_kernel<NT>, dim3(blocks), dim3(NT), 0, s, idx,
                    reinterpret_cast<const uint4*>(x), T, d, E, k, tpb, counts, offsets, src, dest,
                    reinterpret_cast<uint4*>(x_perm), reinterpret_cast<uint2*>(x8), sx, status, fold_cnt, fold_nblk);
}

cudaError_t launch_permute(const int32_t* idx, const __nv_bfloat16* x, int T, int d, int E, int k,
                           int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dest,
                           __nv_bfloat16* x_perm, int32_t* status, int num_sms, cudaStream_t s, uint8_t* x8,
                           float* sx, int32_t* fold_cnt, int fold_nblk) {
    switch (perm_threads(E)) {
        case 1024:
            return launch_permute_nt<1024>(idx, x, T, d, E, k, counts, offsets, src, dest, x_perm, status, num_sms,
                                           s, x8, sx, fold_cnt, fold_nblk);
        case 512:
            return launch_permute_nt<512>(idx, x, T, d, E, k, counts, offsets, src, dest, x_perm, status, num_sms,
                                          s, x8, sx, fold_cnt, fold_nblk);
        default:
            return launch_permute_nt<256>(idx, x, T, d, E, k, counts, offsets, src, dest, x_perm, status, num_sms,
                                          s, x8, sx, fold_cnt, fold_nblk);
    }
}

}  // namespace moe
