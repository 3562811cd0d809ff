// common.cuh — small shared pieces of the MoE kernels (status bits, bf16 packing, launchers).
#pragma once

#include <cuda.h>  // CUtensorMap (type only)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// OR a status bit into the caller's device status word (no-op when none was given).
__device__ __forceinline__ void flag_status(int32_t* status, int32_t bit) {
    if (status) atomicOr(status, bit);
}

// Programmatic dependent launch.  Every kernel of the layer calls pdl_wait() before its first
// global-memory access, which waits for the previous kernel in the stream to finish and its
// writes to become visible (a no-op when the launch had no programmatic dependency); so the
// stream order of all reads and writes is kept, while the launch and the shared-memory /
// tensor-memory set-up of a kernel overlap the tail of the one before.  pdl_trigger() lets the
// next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&v);
}

// Kernels of the layer, as bits of the programmatic-launch mask.
enum PdlKernel { kPdlRoute = 1, kPdlPermute = 2, kPdlGateUp = 4, kPdlDown = 8, kPdlCombine = 16, kPdlQuant = 32 };

// Whether a kernel is launched with the programmatic-stream-serialization attribute (see
// pdl_wait).  The environment variable MOE_PDL, a bit mask of PdlKernel, overrides the default.
bool pdl_enabled(int kernel_bit);
template <typename... KArgs, typename... Args>
cudaError_t launch_k(int kernel_bit, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled(kernel_bit) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Launchers (defined next to their kernels).  All return the launch's error code.
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                         int32_t* status_reset, cudaStream_t s);
cudaError_t launch_route_grouped(const float* logits, const float* bias, int T, int E, int k, int n_group,
                                 int topk_group, float scale, int32_t* idx, float* w, int32_t* status_reset,
                                 cudaStream_t s);
// x8/sx (FP8 layer): when x8 is given, the permuted rows are written as E4M3 codes x8 [T*k, d] with
// a scale per row sx [T*k] (each token quantised once, fp8.cuh) instead of the bf16 x_perm.
cudaError_t launch_permute(const int32_t* idx, const __nv_bfloat16* x, int T, int d, int E, int k,
                           int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dest,
                           __nv_bfloat16* x_perm, int32_t* status, int num_sms, cudaStream_t s,
                           uint8_t* x8 = nullptr, float* sx = nullptr, int32_t* fold_cnt = nullptr,
                           int fold_nblk = 0);
// Steps 1+2 in one launch (softmax router): only when route_permute_fusable(T, E).
bool route_permute_fusable(int T, int E);
cudaError_t launch_route_permute(const float* logits, const __nv_bfloat16* x, int T, int d, int E, int k,
                                 int32_t* idx, float* w, int32_t* counts, int32_t* offsets, int32_t* src,
                                 int32_t* dest, __nv_bfloat16* x_perm, int32_t* status, int num_sms,
                                 cudaStream_t s, uint8_t* x8 = nullptr, float* sx = nullptr,
                                 int32_t* fold_cnt = nullptr, int fold_nblk = 0);
cudaError_t launch_combine(const float* y, const float* w, const int32_t* dest, int T, int d, int k,
                           int ksplit, __nv_bfloat16* out, int32_t* status, cudaStream_t s);

// ---------------------------------------------------------------------------------------------
// Step 5 folded into the down GEMM (moe_forward and moe_forward_fp8 when `cnt` is given).  The
// combine needs all k rows (and K slices) of a token, which different CTAs store at different
// times; instead of a grid-wide barrier each (token, 64-column block) has an arrival counter,
// zeroed by the permute kernel of the same forward.  Every epilogue that has stored its part of
// row r's block b fences its stores and adds its share to counter [src[r], b] (a block's parts
// add up to kFoldWays per row and K slice); the arrival that completes k * ksplit rows folds the
// block: out[t][block] = bf16(sum_j w[t,j] * sum_s y_s[dest[t,j]][block]) in slot and slice order,
// the combine kernel's arithmetic.  No atomics touch the output, so the result is deterministic.
struct FoldArgs {
    int32_t* cnt = nullptr;         // [T, N / kFoldCols] counters; null = no fold (combine launched)
    const int32_t* src = nullptr;   // [M] token of each permuted row
    const int32_t* dest = nullptr;  // [T, k]
    const float* w = nullptr;       // [T, k]
    __nv_bfloat16* out = nullptr;   // [T, N]
    int T = 0, k = 0;
};
constexpr int kFoldCols = 64;
constexpr int kFoldWays = 2;  // arrival units per (row, block, K slice)

// Fold token t's column block b (kFoldCols outputs) from the y_perm slices.
static __device__ __noinline__ void fold_block(const FoldArgs& f, const float* __restrict__ y, long long M, int N,
                                        int ksplit, int t, int b, int32_t* status) {
    __threadfence();  // every arrival's stores before this thread's reads
    const int c0 = b * kFoldCols;
    float acc[kFoldCols];
#pragma unroll
    for (int c = 0; c < kFoldCols; ++c) acc[c] = 0.0f;
    for (int j = 0; j < f.k; ++j) {
        const int r = __ldg(f.dest + static_cast<size_t>(t) * f.k + j);
        if (r < 0 || r >= M) {
            flag_status(status, MOE_STATUS_BAD_DEST);
            continue;
        }
        const float wj = __ldg(f.w + static_cast<size_t>(t) * f.k + j);
        const float* yr = y + static_cast<size_t>(r) * N + c0;
#pragma unroll
        for (int c = 0; c < kFoldCols; c += 4) {
            float4 a = __ldcg(reinterpret_cast<const float4*>(yr + c));
            for (int s = 1; s < ksplit; ++s) {
                const float4 a2 = __ldcg(reinterpret_cast<const float4*>(yr + static_cast<size_t>(s) * M * N + c));
                a.x += a2.x; a.y += a2.y; a.z += a2.z; a.w += a2.w;
            }
            acc[c] += wj * a.x; acc[c + 1] += wj * a.y; acc[c + 2] += wj * a.z; acc[c + 3] += wj * a.w;
        }
    }
    uint4* o = reinterpret_cast<uint4*>(f.out + static_cast<size_t>(t) * N + c0);
#pragma unroll
    for (int c = 0; c < kFoldCols; c += 8)
        o[c / 8] = make_uint4(pack_bf16x2(acc[c], acc[c + 1]), pack_bf16x2(acc[c + 2], acc[c + 3]),
                              pack_bf16x2(acc[c + 4], acc[c + 5]), pack_bf16x2(acc[c + 6], acc[c + 7]));
}

// Row r's part of block b is stored and fenced: count `inc` arrival units; fold if this completes
// the block.
__device__ __forceinline__ void fold_arrive(const FoldArgs& f, const float* y, long long M, int N, int ksplit,
                                            int r, int b, int inc, int32_t* status) {
    const int t = __ldg(f.src + r);
    if (t < 0 || t >= f.T) {
        flag_status(status, MOE_STATUS_BAD_SRC);
        return;
    }
    const int target = kFoldWays * f.k * ksplit;
    const int old = atomicAdd(f.cnt + static_cast<size_t>(t) * (N / kFoldCols) + b, inc);
    if (old + inc == target) fold_block(f, y, M, N, ksplit, t, b, status);
}

// Largest number of K slices the down projection may be split into.
constexpr int kMaxKSplit = 8;

// Grouped GEMMs.  `kind` selects the fused gate+up+SwiGLU (0) or the down projection (1).
struct GemmArgs {
    const void* A;         // x_perm [M,K] bf16 (gate+up) or h [M,K] bf16 (down)
    const void* B;         // W_gate_up [E,K,2N] or W_down [E,K,N], bf16
    const int32_t* offsets;  // [E+1]
    int M, K, N, E;        // N = output features (f for gate+up, d for down)
    void* out;             // h [M,N] bf16, or y_perm [ksplit, M, N] fp32 partial sums
    int32_t* status;
    int ksplit;            // K slices (down only; 1 = no split)
    int swap_max;          // experts with at most this many rows use the swapped orientation
    int pair;              // 0: 1-SM kernel; 1: SM pairs (cta_group::2), normal orientation only;
                           // 2: SM pairs with experts of at most pair_swap_max rows swapped
    int pair_swap_max = 0; // swap threshold of the SM-pair kernel (pair == 2), at most 128
    int pair_layout = 0;   // SM-pair kernel's shared-memory layout: 0 chosen on the device, 1 A, 2 B
    int pair_split = 0;    // SM-pair kernel (pair == 2): CTA pairs given to normal tiles when the
                           // kinds are split between pairs; 0 = one round-robin over all slots
    int inject_stall = 0;  // test hook (1-SM kernel): make one pipeline wait run out, see moe_api.cu
    // Gate+up only: when set, A is x [gather_T, K] and row r of the grouped operand is
    // x[gather_src[r]] (gathered by the kernel); x_perm is never materialised.
    const int32_t* gather_src = nullptr;
    int gather_T = 0;
    // FP8 variant (1-SM kernel): A is [M, K] E4M3 codes with a_scale [M] (one per row), B is
    // [E, N_total, K] E4M3 codes (transposed) with b_scale [E, N_total]; K % 128 == 0.
    bool fp8 = false;
    const float* a_scale = nullptr;
    const float* b_scale = nullptr;
    // Blockwise FP8 (with fp8; launched by launch_grouped_gemm_fp8b): a_scale [M, K/128] (one per
    // 128-wide row block), b_scale [E, N_total/128, K/128] (one per 128 x 128 block), N % 128 == 0.
    bool fp8_blocks = false;
    // Blockwise gate+up only: when set, out receives h's E4M3 codes [M, N] (uint8) and h_scale
    // [M, N/128] the power-of-two scale of each 128-wide block, h quantised in the epilogue.
    float* h_scale = nullptr;
    // Down GEMM only: the combine folded into the epilogue (1-SM and SM-pair kernels; see FoldArgs).
    FoldArgs fold;
};
cudaError_t launch_grouped_gemm(int kind, const GemmArgs& a, int num_sms, cudaStream_t s,
                                const char** why);
cudaError_t launch_grouped_gemm_pair(int kind, const GemmArgs& a, int num_sms, cudaStream_t s,
                                     const char** why);
// Blockwise FP8 (a.fp8_blocks): grouped_gemm_fp8b.cu.
cudaError_t launch_grouped_gemm_fp8b(int kind, const GemmArgs& a, int num_sms, cudaStream_t s, const char** why);

// 2-D bf16 tensor map over [rows, cols] (cols contiguous), box = [box_rows, 64 cols], 128-byte
// swizzle; false if the driver's encoder is unavailable or rejects the operand.
bool make_tensor_map_bf16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                          uint32_t box_rows);
// The same over bytes (FP8 codes): box = [box_rows, 128 cols].
bool make_tensor_map_u8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows);
// Blocked FP8 weight codes (rows x K in 8 KB blocks of 64 rows x 128 K, see moe.h): a box of
// box_rows (a multiple of 64) rows x 128 K codes.
bool make_tensor_map_w8(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows);

// FP8 quantisation (fp8.cu).  Rows: row r of the bf16 [*, C] matrix a (row src[r] when src is
// given, src values checked against src_rows) -> E4M3 codes q [R, C] and scale [R].  Weights:
// W [E, K, N] bf16 -> Wq codes, transposed and blocked ([E, N/64, K/128, 64, 128]: code (e, n, k) at
// [e][n / 64][k / 128][n % 64][k % 128]), and scale [E, N], one per output column.
cudaError_t launch_quantize_rows_fp8(const __nv_bfloat16* a, const int32_t* src, int R, int C, int src_rows,
                                     uint8_t* q, float* scale, int32_t* status, cudaStream_t s);
cudaError_t launch_quantize_weights_fp8(const __nv_bfloat16* W, int E, int K, int N, uint8_t* Wq, float* scale,
                                        cudaStream_t s);
// Blockwise FP8 (fp8.cu): 128-wide row blocks (scale [R, C/128]) and 128 x 128 weight blocks
// (scale [E, N/128, K/128]; codes in the same blocked layout), power-of-two scales.
cudaError_t launch_quantize_rows_fp8b(const __nv_bfloat16* a, const int32_t* src, int R, int C, int src_rows,
                                      uint8_t* q, float* scale, int32_t* status, cudaStream_t s);
cudaError_t launch_quantize_weights_fp8b(const __nv_bfloat16* W, int E, int K, int N, uint8_t* Wq, float* scale,
                                         cudaStream_t s);

}  // namespace moe
