// combine.cu — step 5: weighted combine / unpermute,
//   out[t] = bf16( sum_{j=0..k-1} w[t,j] * y_perm[dest[t,j]] ),  fp32 sums in slot order.
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

__global__ void __launch_bounds__(kCombThreads)
combine_kernel(const float4* __restrict__ y, const float* __restrict__ w,
               const int32_t* __restrict__ dest, int T, int d, int k, uint4* __restrict__ out,
               int32_t* __restrict__ status) {
    __shared__ int rows[kMaxK];
    __shared__ float wts[kMaxK];
    const int t = blockIdx.x, tid = threadIdx.x;
    const long long M = static_cast<long long>(T) * k;
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
            const float4 a = __ldg(yr), b = __ldg(yr + 1);
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
                           __nv_bfloat16* out, int32_t* status, cudaStream_t s) {
    combine_kernel<<<T, kCombThreads, 0, s>>>(reinterpret_cast<const float4*>(y), w, dest, T, d, k,
                                              reinterpret_cast<uint4*>(out), status);
    return cudaGetLastError();
}

}  // namespace moe
