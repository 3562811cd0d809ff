// combine.cu — step 5: weighted combine / unpermute,
//   out[t] = bf16( sum_{j=0..k-1} w[t,j] * y_perm[dest[t,j]] ),  fp32 sums in slot order.
// When the down projection was split over K, y_perm holds `ksplit` partial slices [ksplit, T*k, d]
// and each row is first summed over the slices in slice order (a fixed order: deterministic).
// DeepGEMM PR #304 write-up, section 1.1 ("combine"); HPC-Ops page, FusedMoE paragraph (the
// weighted-average reduce after the GroupGEMM).
//
// Gather form: block (t, c) owns a set of token t's output columns (every gridDim.y-th group of
// 1024) and reads those columns of the token's k rows, so no two blocks write the same output and
// no atomics are needed — the result is deterministic.  Each thread owns 8 outputs at a time: it
// issues all k slots' 2 x 16-byte fp32 loads before adding them in slot order, then one 16-byte
// bf16 store; accesses are coalesced across the block.  Few tokens split their columns over
// several blocks so that enough loads are in flight (T=32: 128 blocks instead of 32); many tokens
// use one block each (T=4096: 4096 blocks of 4 column groups rather than 16384 blocks of one).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kCombThreads = 128;
constexpr int kMaxK = 8;

// SPLIT = y_perm holds more than one K slice (kept a template so the common single-slice case
// has no inner loop between the slot loads).
// KB = slots held in registers at once (k <= KB): sized to k so that a top-2 layer does not
// reserve registers for eight slots (which would cost occupancy).
template <bool SPLIT, int KB>
__global__ void __launch_bounds__(kCombThreads)
combine_kernel(const float4* __restrict__ y, const float* __restrict__ w,
               const int32_t* __restrict__ dest, int T, int d, int k, int ksplit, uint4* __restrict__ out,
               int32_t* __restrict__ status) {
    __shared__ int rows[kMaxK];
    __shared__ float wts[kMaxK];
    const int t = blockIdx.x, tid = threadIdx.x;
    const long long M = static_cast<long long>(T) * k;
    pdl_wait();
    pdl_trigger();
    if (tid < k) {
        const int r = __ldg(dest + static_cast<size_t>(t) * k + tid);
        const bool ok = r >= 0 && r < M;
        if (!ok) flag_status(status, MOE_STATUS_BAD_DEST);
        rows[tid] = ok ? r : -1;
        wts[tid] = __ldg(w + static_cast<size_t>(t) * k + tid);
    }
    __syncthreads();

    const int dv = d / 8;  // groups of 8 outputs
    for (int v = blockIdx.y * kCombThreads + tid; v < dv; v += gridDim.y * kCombThreads) {
        float4 a[KB], b[KB];
#pragma unroll
        for (int j = 0; j < KB; ++j)
            if (j < k && rows[j] >= 0) {
                const float4* yr = y + static_cast<size_t>(rows[j]) * (d / 4) + 2 * v;
                a[j] = __ldg(yr);
                b[j] = __ldg(yr + 1);
                if (SPLIT)
                    for (int s = 1; s < ksplit; ++s) {
                        const float4* ys = yr + static_cast<size_t>(s) * M * (d / 4);
                        const float4 a2 = __ldg(ys), b2 = __ldg(ys + 1);
                        a[j].x += a2.x; a[j].y += a2.y; a[j].z += a2.z; a[j].w += a2.w;
                        b[j].x += b2.x; b[j].y += b2.y; b[j].z += b2.z; b[j].w += b2.w;
                    }
            }
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < KB; ++j)
            if (j < k && rows[j] >= 0) {
                const float wj = wts[j];
                acc[0] += wj * a[j].x; acc[1] += wj * a[j].y; acc[2] += wj * a[j].z; acc[3] += wj * a[j].w;
                acc[4] += wj * b[j].x; acc[5] += wj * b[j].y; acc[6] += wj * b[j].z; acc[7] += wj * b[j].w;
            }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        out[static_cast<size_t>(t) * dv + v] = o;
    }
}

}  // namespace

cudaError_t launch_combine(const float* y, const float* w, const int32_t* dest, int T, int d, int k,
                           int ksplit, __nv_bfloat16* out, int32_t* status, cudaStream_t s) {
    auto kernel = k <= 2 ? (ksplit > 1 ? combine_kernel<true, 2> : combine_kernel<false, 2>)
                : k <= 4 ? (ksplit > 1 ? combine_kernel<true, 4> : combine_kernel<false, 4>)
                         : (ksplit > 1 ? combine_kernel<true, 8> : combine_kernel<false, 8>);
    // Column groups per token: enough blocks for ~4 per SM on a 152-SM GPU, at most one per
    // 1024-column group.
    const int groups = (d / 8 + kCombThreads - 1) / kCombThreads;
    int split = (4 * 152 + T - 1) / T;
    split = split < 1 ? 1 : (split > groups ? groups : split);
    const dim3 grid(T, split);
    return launch_k(kPdlCombine, kernel, grid, dim3(kCombThreads), 0, s, reinterpret_cast<const float4*>(y), w,
                    dest, T, d, k, ksplit, reinterpret_cast<uint4*>(out), status);
}

}  // namespace moe
