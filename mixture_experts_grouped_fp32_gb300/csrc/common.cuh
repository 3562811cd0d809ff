// common.cuh — small shared pieces of the MoE kernels (status bits, bf16 packing, launchers).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// OR a status bit into the caller's device status word (no-op when none was given).
__device__ __forceinline__ void flag_status(int32_t* status, int32_t bit) {
    if (status) atomicOr(status, bit);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&v);
}

// Launchers (defined next to their kernels).  All return cudaGetLastError() of the launch.
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                         int32_t* status_reset, cudaStream_t s);
cudaError_t launch_permute(const int32_t* idx, const __nv_bfloat16* x, int T, int d, int E, int k,
                           int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dest,
                           __nv_bfloat16* x_perm, int32_t* status, int num_sms, cudaStream_t s);
cudaError_t launch_combine(const float* y, const float* w, const int32_t* dest, int T, int d, int k,
                           __nv_bfloat16* out, int32_t* status, cudaStream_t s);

// Grouped GEMMs.  `kind` selects the fused gate+up+SwiGLU (0) or the down projection (1).
struct GemmArgs {
    const void* A;         // x_perm [M,K] bf16 (gate+up) or h [M,K] bf16 (down)
    const void* B;         // W_gate_up [E,K,2N] or W_down [E,K,N], bf16
    const int32_t* offsets;  // [E+1]
    int M, K, N, E;        // N = output features (f for gate+up, d for down)
    void* out;             // h [M,N] bf16 or y_perm [M,N] fp32
    int32_t* status;
};
cudaError_t launch_grouped_gemm(int kind, const GemmArgs& a, int num_sms, cudaStream_t s,
                                const char** why);

}  // namespace moe
