// combine.cu — step 5: weighted combine / unpermute,
//   out[t] = bf16( sum_{j=0..k-1} w[t,j] * y_perm[dest[t,j]] ),  fp32 sums in slot order.
// When the down projection was split over K, y_perm holds `ksplit` partial slices [ksplit, T*k, d]
// and each row is first summed over the slices in slice order (a fixed order: deterministic).
// DeepGEMM PR #304 write-up, section 1.1 ("combine"); HPC-Ops page, FusedMoE paragraph (the
// weighted-average reduce after the GroupGEMM).
//
// Gather form: each block owns one token and reads its k rows, so no two blocks write the same
// output and no atomics are needed — the result is deterministic.  Accesses are 2 x 16-byte fp32
// loads per slot and one 16-byte bf16 store per 8 output elements, coalesced across the block.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kCombThreads = 128;
constexpr int kMaxK = 8;

// SPLIT = y_perm holds more than one K slice (kept a template so the common single-slice case
// has no inner loop between the slot loads).
template <bool SPLIT>
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
    for (int v = tid; v < dv; v += kCombThreads) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
            const int r = rows[j];
            if (r < 0) continue;
            const float wj = wts[j];
            const float4* yr = y + static_cast<size_t>(r) * (d / 4) + 2 * v;
            float4 a = __ldg(yr), b = __ldg(yr + 1);
            if (SPLIT)
            for (int s = 1; s < ksplit; ++s) {
                const float4* ys = yr + static_cast<size_t>(s) * M * (d / 4);
                const float4 a2 = __ldg(ys), b2 = __ldg(ys + 1);
                a.x += a2.x; a.y += a2.y; a.z += a2.z; a.w += a2.w;
                b.x += b2.x; b.y += b2.y; b.z += b2.z; b.w += b2.w;
            }
            acc[0] += wj * a.x; acc[1] += wj * a.y; acc[2] += wj * a.z; acc[3] += wj * a.w;
            acc[4] += wj * b.x; acc[5] += wj * b.y; acc[6] += wj * b.z; acc[7] += wj * b.w;
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
    auto kernel = ksplit > 1 ? combine_kernel<true> : combine_kernel<false>;
    return launch_k(kPdlCombine, kernel, dim3(T), dim3(kCombThreads), 0, s, reinterpret_cast<const float4*>(y), w,
                    dest, T, d, k, ksplit, reinterpret_cast<uint4*>(out), status);
}

}  // namespace moe
