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

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;  // tokens per 256-thread block
constexpr int kMaxK = 8;

// Does candidate (av, ai) rank before (bv, bi)?  Larger logit first, lower id on equal logits;
// id INT_MAX marks "no candidate".
__device__ __forceinline__ bool ranks_before(float av, int ai, float bv, int bi) {
    if (ai == INT_MAX) return false;
    if (bi == INT_MAX) return true;
    return av > bv || (av == bv && ai < bi);
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
            // Butterfly arg-max: ranks_before is a strict total order on distinct ids, so every
            // lane ends with the same winner.
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

}  // namespace

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
