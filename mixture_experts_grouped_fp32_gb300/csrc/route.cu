// route.cu — step 1: top-k routing with softmax-renormalised weights, one warp per token.
//
// Routing happens on the device with no host synchronisation ("Triton MoE 核心擊敗 Megablocks",
// setupai.cc, section 技術深入, dynamic-routing bullet).  The pages leave the router function
// open; the reading used is: the k largest fp32 logits (equal logits -> lower expert id first,
// slots ordered by descending logit), weights = softmax over all experts restricted to those k
// and renormalised, which equals exp(l_j - l_max) / sum_j' exp(l_j' - l_max) over the chosen j.
// Selection compares the fp32 logits themselves, so the chosen ids do not depend on how exp()
// rounds and match a CPU reference bit for bit.
#include <climits>
#include <cmath>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;  // tokens per 256-thread block
constexpr int kMaxK = 8;

// Does candidate (av, ai) rank before (bv, bi)?  Larger logit first, lower id on equal logits;
// id INT_MAX marks "no candidate".  A NaN ranks below every number (NaNs among themselves by id),
// so the order stays total and no expert can win two slots of one token.
__device__ __forceinline__ bool ranks_before(float av, int ai, float bv, int bi) {
    if (ai == INT_MAX) return false;
    if (bi == INT_MAX) return true;
    const bool an = av != av, bn = bv != bv;
    if (an != bn) return bn;
    return av > bv || ((av == bv || an) && ai < bi);
}

// EPL = experts held per lane (ceil(E / 32)), expert e lives in lane e % 32, register e / 32.
template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ idx,
             float* __restrict__ w, int32_t* __restrict__ status_reset) {
    pdl_wait();
    pdl_trigger();
    if (status_reset != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *status_reset = 0;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
    if (t >= T) return;  // whole warp leaves together

    const float* row = logits + static_cast<size_t>(t) * E;
    float v[EPL];
    bool avail[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        avail[i] = e < E;
        v[i] = avail[i] ? __ldg(row + e) : 0.0f;
    }

    float sel_v[kMaxK];
    int sel_i[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
        sel_v[j] = 0.0f;
        sel_i[j] = 0;
        if (j < k) {
            float bv = 0.0f;
            int bi = INT_MAX;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (avail[i] && ranks_before(v[i], lane + 32 * i, bv, bi)) {
                    bv = v[i];
                    bi = lane + 32 * i;
                }
            // Butterfly arg-max: ranks_before is a strict total order on distinct ids (NaN
            // included), so every lane ends with the same winner.
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ranks_before(ov, oi, bv, bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (lane + 32 * i == bi) avail[i] = false;
            sel_v[j] = bv;
            sel_i[j] = bi;
        }
    }

    // Softmax restricted to the chosen experts; slot 0 holds the largest logit.
    float ex[kMaxK];
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
        ex[j] = 0.0f;
        if (j < k) {
            ex[j] = expf(sel_v[j] - sel_v[0]);
            s += ex[j];
        }
    }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
        if (j < k && lane == j) {
            idx[static_cast<size_t>(t) * k + j] = sel_i[j];
            w[static_cast<size_t>(t) * k + j] = ex[j] / s;
        }
}

// ---------------------------------------------------------------------------------------------
// DeepSeek-V3's router (DeepSeek-V3 Technical Report, section 2.1.2): affinity s = sigmoid(logit);
// the selection score c = s + bias (the auxiliary-loss-free balancing bias steers the choice only);
// the E experts form n_group equal groups, a group's score is the sum of its q = k / topk_group
// largest c (the report's node-limited routing: the sum of the highest K_r / M scores per node);
// the topk_group best groups are kept (equal scores -> lower group) and the k largest c among their
// experts are chosen (equal -> lower id; slot order = descending c); w = scale * s / sum of the
// chosen s (summed in slot order).  All comparisons are on the fp32 values themselves.
// ---------------------------------------------------------------------------------------------
constexpr int kMaxGroups = 32;

// GS32: every group is exactly 32 experts (E = 32 * n_group, so group g = register g of every lane)
// and q <= 2 — DeepSeek-V3's shape.  Then one butterfly pass merges the per-lane top-2 of all
// groups at once and the group scores stay in registers.
template <int EPL, bool GS32>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_grouped_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k,
                     int n_group, int topk_group, float scale, int32_t* __restrict__ idx,
                     float* __restrict__ w, int32_t* __restrict__ status_reset) {
    pdl_wait();
    pdl_trigger();
    if (status_reset != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *status_reset = 0;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
    if (t >= T) return;  // whole warp leaves together

    const int gs = E / n_group;
    const int q = min(gs, max(1, k / topk_group));
    const float* row = logits + static_cast<size_t>(t) * E;
    float s[EPL], c[EPL];
    int grp[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        s[i] = 0.0f;
        c[i] = 0.0f;
        grp[i] = -1;  // -1: no expert in this register
        if (e < E) {
            s[i] = 1.0f / (1.0f + expf(-__ldg(row + e)));
            c[i] = s[i] + __ldg(bias + e);
            grp[i] = e / gs;
        }
    }

    unsigned kept = 0u;
    if (GS32) {
        // Top-2 of each register across the warp: merge sorted pairs (a1 >= a2), (b1 >= b2) into
        // max(a1, b1) >= max(min(a1, b1), max(a2, b2)).
        float t1[EPL], t2[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            t1[i] = c[i];
            t2[i] = -INFINITY;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const float o1 = __shfl_xor_sync(0xffffffffu, t1[i], off);
                const float o2 = __shfl_xor_sync(0xffffffffu, t2[i], off);
                const float hi = fmaxf(t1[i], o1), lo = fminf(t1[i], o1);
                t2[i] = fmaxf(lo, fmaxf(t2[i], o2));
                t1[i] = hi;
            }
        }
        float gs_reg[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) gs_reg[i] = q == 1 ? 0.0f + t1[i] : (0.0f + t1[i]) + t2[i];
        for (int r = 0; r < topk_group; ++r) {
            int bg = -1;
            float bv = 0.0f;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (i < n_group && !(kept & (1u << i)) && (bg < 0 || gs_reg[i] > bv)) {
                    bg = i;
                    bv = gs_reg[i];
                }
            kept |= 1u << bg;
        }
    } else {
    // Group scores: q rounds of a warp arg-max per group, adding the winners largest first.
    float gscore[kMaxGroups];
    for (int g = 0; g < n_group; ++g) {
        unsigned taken = 0u;  // this lane's registers already counted for group g
        float sum = 0.0f;
        for (int r = 0; r < q; ++r) {
            float bv = 0.0f;
            int bi = INT_MAX;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (grp[i] == g && !(taken & (1u << i)) && ranks_before(c[i], lane + 32 * i, bv, bi)) {
                    bv = c[i];
                    bi = lane + 32 * i;
                }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ranks_before(ov, oi, bv, bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (lane + 32 * i == bi) taken |= 1u << i;
            sum += bv;
        }
        gscore[g] = sum;  // identical in every lane
    }

    // Keep the topk_group best groups (every lane takes the same decisions).
    for (int r = 0; r < topk_group; ++r) {
        int bg = -1;
        for (int g = 0; g < n_group; ++g)
            if (!(kept & (1u << g)) && (bg < 0 || gscore[g] > gscore[bg])) bg = g;
        kept |= 1u << bg;
    }
    }

    // The k largest selection scores among the kept groups' experts.
    bool avail[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) avail[i] = grp[i] >= 0 && (kept & (1u << grp[i]));
    float sel_s[kMaxK];
    int sel_i[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
        sel_s[j] = 0.0f;
        sel_i[j] = 0;
        if (j < k) {
            float bv = 0.0f, bs = 0.0f;
            int bi = INT_MAX;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (avail[i] && ranks_before(c[i], lane + 32 * i, bv, bi)) {
                    bv = c[i];
                    bs = s[i];
                    bi = lane + 32 * i;
                }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const float os = __shfl_xor_sync(0xffffffffu, bs, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ranks_before(ov, oi, bv, bi)) {
                    bv = ov;
                    bs = os;
                    bi = oi;
                }
            }
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (lane + 32 * i == bi) avail[i] = false;
            sel_s[j] = bs;
            sel_i[j] = bi;
        }
    }
    float ssum = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
        if (j < k) ssum += sel_s[j];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
        if (j < k && lane == j) {
            idx[static_cast<size_t>(t) * k + j] = sel_i[j];
            w[static_cast<size_t>(t) * k + j] = scale * (sel_s[j] / ssum);
        }
}

}  // namespace

cudaError_t launch_route_grouped(const float* logits, const float* bias, int T, int E, int k, int n_group,
                                 int topk_group, float scale, int32_t* idx, float* w, int32_t* status_reset,
                                 cudaStream_t s) {
    const dim3 grid((T + kRouteWarps - 1) / kRouteWarps), block(kRouteWarps * 32);
    const int q = min(E / n_group, max(1, k / topk_group));
    const bool gs32 = E == 32 * n_group && q <= 2;
#define MOE_ROUTE_GROUPED(EPL, GS)                                                                        \
    launch_k(kPdlRoute, route_grouped_kernel<EPL, GS>, grid, block, 0, s, logits, bias, T, E, k, n_group, \
             topk_group, scale, idx, w, status_reset)
    if (gs32) {
        if (E == 32) return MOE_ROUTE_GROUPED(1, true);
        if (E == 64) return MOE_ROUTE_GROUPED(2, true);
        if (E == 128) return MOE_ROUTE_GROUPED(4, true);
        if (E == 256) return MOE_ROUTE_GROUPED(8, true);
    }
    if (E <= 32) return MOE_ROUTE_GROUPED(1, false);
    if (E <= 64) return MOE_ROUTE_GROUPED(2, false);
    if (E <= 128) return MOE_ROUTE_GROUPED(4, false);
    return MOE_ROUTE_GROUPED(8, false);
#undef MOE_ROUTE_GROUPED
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                         int32_t* status_reset, cudaStream_t s) {
    const dim3 grid((T + kRouteWarps - 1) / kRouteWarps), block(kRouteWarps * 32);
    if (E <= 32)
        return launch_k(kPdlRoute, route_kernel<1>, grid, block, 0, s, logits, T, E, k, idx, w, status_reset);
    else if (E <= 64)
        return launch_k(kPdlRoute, route_kernel<2>, grid, block, 0, s, logits, T, E, k, idx, w, status_reset);
    else if (E <= 128)
        return launch_k(kPdlRoute, route_kernel<4>, grid, block, 0, s, logits, T, E, k, idx, w, status_reset);
    else
        return launch_k(kPdlRoute, route_kernel<8>, grid, block, 0, s, logits, T, E, k, idx, w, status_reset);
}

}  // namespace moe
