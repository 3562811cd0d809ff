// fp8.cu — FP8 (E4M3) quantisation for the FP8 variant of the layer's grouped GEMMs.
//
// Scaling: per row for activations (each x_perm row, each h row), per output channel for the
// weights (expert e, output column n, over K): absmax over the row / channel, inv = 448 / absmax,
// code = E4M3(value * inv) rounded to nearest even with saturation, dequantisation scale =
// absmax / 448 (an all-zero row: scale 1, zero codes).  These scales factor out of every dot
// product, so the FP8 GEMMs accumulate decoded codes in fp32 and apply scale_row * scale_col in
// their epilogue.  DeepGEMM PR #304 write-up, section 5.3 (an FP8 grouped GEMM on SM100) and its
// Mega MoE epilogue (SwiGLU then FP8 quantisation) are the pages' FP8 context; their 128-wide
// blockwise scales are not used here (they need per-K-block promotion of the accumulator).
#include "common.cuh"
#include "fp8.cuh"

namespace moe {
namespace {

constexpr int kQThreads = 256;

// Block-wide max of non-negative floats (every thread gets the result).
__device__ __forceinline__ float block_max(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();  // red may still be read from a previous call
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float m = 0.0f;
    for (int i = 0; i < kQThreads / 32; ++i) m = fmaxf(m, red[i]);
    return m;
}

// One block per output row r: source row src[r] (or r when src is null) of a bf16 matrix with C
// columns (C % 8 == 0) -> codes [r, C] and scale[r].
__global__ void __launch_bounds__(kQThreads)
quantize_rows_kernel(const uint4* __restrict__ a, const int32_t* __restrict__ src, int R, int C, int src_rows,
                     uint2* __restrict__ q, float* __restrict__ scale, int32_t* __restrict__ status) {
    __shared__ float red[kQThreads / 32];
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x;
    if (r >= R) return;
    int s = src ? __ldg(src + r) : r;
    if (s < 0 || s >= src_rows) {  // bad src: a zero row, reported
        flag_status(status, MOE_STATUS_BAD_SRC);
        s = -1;
    }
    const int cv = C / 8;  // uint4 (8 bf16) per row
    const uint4* row = a + static_cast<size_t>(s < 0 ? 0 : s) * cv;
    float m = 0.0f;
    if (s >= 0)
        for (int v = threadIdx.x; v < cv; v += kQThreads) m = fmaxf(m, absmax8(__ldg(row + v)));
    const float amax = block_max(m, red);
    const float inv = fp8_inv(amax);
    if (threadIdx.x == 0) scale[r] = fp8_scale(amax);
    uint2* out = q + static_cast<size_t>(r) * cv;
    for (int v = threadIdx.x; v < cv; v += kQThreads) {
        uint4 p = make_uint4(0, 0, 0, 0);
        if (s >= 0) p = __ldg(row + v);
        out[v] = codes8(p, inv);
    }
}

// Weights W [E, K, N] bf16 -> Wq blocked codes (code (e, n, k) at [e][n / 64][k / 128][n % 64]
// [k % 128]: 8 KB blocks of 64 output columns x 128 K) and scale [E, N]; block (e, 64-column group).
// Pass 1: per-column absmax over K.  Pass 2: 64 x 64 tiles transposed through shared memory, so
// reads (64 columns of a K-row) and writes (64 K-bytes of an output row) are both contiguous.
constexpr int kWCols = 64;
__global__ void __launch_bounds__(kQThreads)
quantize_weights_kernel(const uint16_t* __restrict__ W, int K, int N, uint8_t* __restrict__ Wq,
                        float* __restrict__ scale) {
    __shared__ float cmax[kQThreads / kWCols][kWCols];
    __shared__ float inv[kWCols];
    __shared__ uint8_t tile[kWCols][kWCols + 4];
    const int e = blockIdx.y, n0 = blockIdx.x * kWCols;
    const int c = threadIdx.x % kWCols, rr = threadIdx.x / kWCols;  // 4 row phases x 64 columns
    const uint16_t* We = W + static_cast<size_t>(e) * K * N;
    const bool col_ok = n0 + c < N;
    float m = 0.0f;
    if (col_ok)
        for (int k = rr; k < K; k += kQThreads / kWCols)
            m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(__ldg(We + static_cast<size_t>(k) * N + n0 + c)) << 16)));
    cmax[rr][c] = m;
    __syncthreads();
    if (threadIdx.x < kWCols) {
        float a = 0.0f;
        for (int i = 0; i < kQThreads / kWCols; ++i) a = fmaxf(a, cmax[i][threadIdx.x]);
        inv[threadIdx.x] = fp8_inv(a);
        if (n0 + static_cast<int>(threadIdx.x) < N) scale[static_cast<size_t>(e) * N + n0 + threadIdx.x] = fp8_scale(a);
    }
    __syncthreads();
    // This block's 64 columns form one 64-row group of the blocked layout: K / 128 blocks of 8 KB.
    uint8_t* Wqg = Wq + static_cast<size_t>(e) * N * K + static_cast<size_t>(n0) * K;
    for (int k0 = 0; k0 < K; k0 += kWCols) {
        for (int i = threadIdx.x; i < kWCols * kWCols; i += kQThreads) {
            const int kk = i / kWCols, cc = i % kWCols;  // read: row k0+kk, column n0+cc
            uint8_t code = 0;
            if (k0 + kk < K && n0 + cc < N)
                code = to_e4m3(__uint_as_float(static_cast<uint32_t>(__ldg(We + static_cast<size_t>(k0 + kk) * N + n0 + cc)) << 16) * inv[cc]);
            tile[cc][kk] = code;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kWCols * kWCols; i += kQThreads) {
            const int cc = i / kWCols, kk = i % kWCols;  // write: output row n0+cc, K-byte k0+kk
            const int k = k0 + kk;
            if (k < K && n0 + cc < N) Wqg[static_cast<size_t>(k >> 7) * 8192 + cc * 128 + (k & 127)] = tile[cc][kk];
        }
        __syncthreads();
    }
}

// The same quantisation of W [E, K, N] bf16 (16-byte aligned; N % 64 == 0, K % 128 == 0) in three
// steps with 16-byte loads.  1) Column maxima over K chunks: CTA (256 columns, 256 K rows, e), a
// thread 8 columns of every 8th row, the chunk's maxima merged into colmax[e][n] (zeroed first) by
// an integer atomicMax on the float bits, which orders non-negative floats as floats.
constexpr int kCmCols = 256, kCmRows = 256;
__global__ void __launch_bounds__(kQThreads)
weights_colmax_kernel(const uint4* __restrict__ W, int K, int N, unsigned int* __restrict__ colmax) {
    __shared__ float red[kQThreads / 32][kCmCols];
    const int e = blockIdx.z, n0 = blockIdx.x * kCmCols, k0 = blockIdx.y * kCmRows;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // column group, row phase
    const int c8 = n0 + 8 * tx;
    float m[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    if (c8 < N) {
        const int k1 = min(K, k0 + kCmRows);
        const uint4* col = W + (static_cast<size_t>(e) * K * N + c8) / 8;
        for (int k = k0 + ty; k < k1; k += kQThreads / 32) {
            const uint4 p = __ldg(col + static_cast<size_t>(k) * (N / 8));
            const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                m[2 * i] = fmaxf(m[2 * i], fabsf(bf16_lo(w[i])));
                m[2 * i + 1] = fmaxf(m[2 * i + 1], fabsf(bf16_hi(w[i])));
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) red[ty][8 * tx + i] = m[i];
    __syncthreads();
    const int c = threadIdx.x;  // one column of the CTA's 256
    if (n0 + c < N) {
        float a = 0.0f;
#pragma unroll
        for (int r = 0; r < kQThreads / 32; ++r) a = fmaxf(a, red[r][c]);
        atomicMax(colmax + static_cast<size_t>(e) * N + n0 + c, __float_as_uint(a));
    }
}

// 2) One 8 KB output block per CTA (64 output columns x 128 K of expert e): the 128 x 64 tile read
// row by row (16-byte loads), converted with its columns' 448 / max, transposed through shared
// memory and written as 64 contiguous 128-byte rows.
__global__ void __launch_bounds__(kQThreads)
weights_tile_kernel(const uint4* __restrict__ W, int K, int N, const float* __restrict__ colmax,
                    uint8_t* __restrict__ Wq) {
    __shared__ float inv[64];
    __shared__ __align__(16) uint8_t tile[64][128 + 16];
    const int e = blockIdx.z, n0 = blockIdx.x * 64, k0 = blockIdx.y * 128;
    if (threadIdx.x < 64) inv[threadIdx.x] = fp8_inv(colmax[static_cast<size_t>(e) * N + n0 + threadIdx.x]);
    __syncthreads();
    const uint4* src = W + (static_cast<size_t>(e) * K * N + static_cast<size_t>(k0) * N + n0) / 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // 128 rows x 8 uint4 = 1024 loads, 4 a thread
        const int v = threadIdx.x + j * kQThreads, kk = v >> 3, g = v & 7;
        const uint4 p = __ldg(src + static_cast<size_t>(kk) * (N / 8) + g);
        const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            tile[8 * g + 2 * i][kk] = to_e4m3(bf16_lo(w[i]) * inv[8 * g + 2 * i]);
            tile[8 * g + 2 * i + 1][kk] = to_e4m3(bf16_hi(w[i]) * inv[8 * g + 2 * i + 1]);
        }
    }
    __syncthreads();
    uint8_t* dst = Wq + static_cast<size_t>(e) * N * K + static_cast<size_t>(n0) * K + static_cast<size_t>(k0 >> 7) * 8192;
#pragma unroll
    for (int j = 0; j < 2; ++j) {  // 512 uint4 of output, 2 a thread
        const int v = threadIdx.x + j * kQThreads, c = v >> 3, q = v & 7;
        reinterpret_cast<uint4*>(dst)[v] = *reinterpret_cast<const uint4*>(&tile[c][16 * q]);
    }
}

// 3) Column maxima -> scales in place.
__global__ void __launch_bounds__(kQThreads)
colmax_to_scale_kernel(float* __restrict__ scale, int n) {
    const int i = blockIdx.x * kQThreads + threadIdx.x;
    if (i < n) scale[i] = fp8_scale(scale[i]);
}

// Blockwise rows: one CTA per output row r (source row src[r], or r), 128-wide blocks of C
// (C % 128 == 0) -> codes and one power-of-two scale per block, scale [R, C/128].  Half a warp per
// block (16 lanes x 8 values); a warp takes two blocks at a time.
__global__ void __launch_bounds__(kQThreads)
quantize_rows_blocks_kernel(const uint4* __restrict__ a, const int32_t* __restrict__ src, int R, int C,
                            int src_rows, uint2* __restrict__ q, float* __restrict__ scale,
                            int32_t* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x;
    if (r >= R) return;
    int s = src ? __ldg(src + r) : r;
    if (s < 0 || s >= src_rows) {  // bad src: a zero row, reported
        if (threadIdx.x == 0) flag_status(status, MOE_STATUS_BAD_SRC);
        s = -1;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cv = C / 8, nblk = C / 128;
    const uint4* row = a + static_cast<size_t>(s < 0 ? 0 : s) * cv;
    for (int bp = warp; bp < (nblk + 1) / 2; bp += kQThreads / 32) {  // warp-uniform trip count
        const int b = 2 * bp + (lane >> 4);
        const bool valid = b < nblk;
        const int v = b * 16 + (lane & 15);
        uint4 p = make_uint4(0, 0, 0, 0);
        if (valid && s >= 0) p = __ldg(row + v);
        float m = absmax8(p);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));  // within 16 lanes
        const float P = pow2_block_scale(m);
        if (valid) {
            q[static_cast<size_t>(r) * cv + v] = codes8(p, 1.0f / P);
            if ((lane & 15) == 0) scale[static_cast<size_t>(r) * nblk + b] = P;
        }
    }
}

// Blockwise weights: W [E, K, N] bf16 -> blocked codes (as quantize_weights_kernel) and one
// power-of-two scale per 128 x 128 block of (output column, K), scale [E, N/128, K/128].  CTA
// (n block, k block, e): the block through shared memory, its absmax, then 64 codes per thread
// (one output column, half of the K block) written as 64 contiguous bytes.
constexpr int kWB = 128;
__global__ void __launch_bounds__(kQThreads)
quantize_weights_blocks_kernel(const uint16_t* __restrict__ W, int K, int N, uint8_t* __restrict__ Wq,
                               float* __restrict__ scale) {
    __shared__ uint16_t tile[kWB][kWB + 2];  // [k][n], padded against bank conflicts in the column reads
    __shared__ float red[kQThreads / 32];
    const int nb = blockIdx.x, kb = blockIdx.y, e = blockIdx.z;
    const uint16_t* We = W + static_cast<size_t>(e) * K * N;
    float m = 0.0f;
    for (int i = threadIdx.x; i < kWB * kWB / 2; i += kQThreads) {  // bf16 pairs
        const int k = i / (kWB / 2), n2 = i % (kWB / 2);
        const uint32_t w2 = __ldg(reinterpret_cast<const uint32_t*>(We + static_cast<size_t>(kb * kWB + k) * N + nb * kWB) + n2);
        tile[k][2 * n2] = static_cast<uint16_t>(w2 & 0xFFFFu);
        tile[k][2 * n2 + 1] = static_cast<uint16_t>(w2 >> 16);
        m = fmaxf(m, fmaxf(fabsf(bf16_lo(w2)), fabsf(bf16_hi(w2))));
    }
    const float amax = block_max(m, red);
    const float P = pow2_block_scale(amax), inv = 1.0f / P;
    if (threadIdx.x == 0) scale[(static_cast<size_t>(e) * (N / kWB) + nb) * (K / kWB) + kb] = P;
    __syncthreads();
    const int n = threadIdx.x >> 1, k0 = (threadIdx.x & 1) * 64;  // output column, K half
    const int gn = nb * kWB + n;
    uint8_t* dst = Wq + static_cast<size_t>(e) * N * K + static_cast<size_t>(gn >> 6) * K * 64 +
                   static_cast<size_t>(kb) * 8192 + (gn & 63) * 128 + k0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {  // 4 x 16 codes
        uint32_t o[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float v = __uint_as_float(static_cast<uint32_t>(tile[k0 + c * 16 + j][n]) << 16) * inv;
            o[j >> 2] |= static_cast<uint32_t>(to_e4m3(v)) << (8 * (j & 3));
        }
        reinterpret_cast<uint4*>(dst)[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_quantize_rows_fp8b(const __nv_bfloat16* a, const int32_t* src, int R, int C, int src_rows,
                                      uint8_t* q, float* scale, int32_t* status, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    return launch_k(kPdlQuant, quantize_rows_blocks_kernel, dim3(R), dim3(kQThreads), 0, s,
                    reinterpret_cast<const uint4*>(a), src, R, C, src_rows, reinterpret_cast<uint2*>(q), scale,
                    status);
}

cudaError_t launch_quantize_weights_fp8b(const __nv_bfloat16* W, int E, int K, int N, uint8_t* Wq, float* scale,
                                         cudaStream_t s) {
    const dim3 grid(N / kWB, K / kWB, E);
    quantize_weights_blocks_kernel<<<grid, kQThreads, 0, s>>>(reinterpret_cast<const uint16_t*>(W), K, N, Wq, scale);
    return cudaGetLastError();
}

cudaError_t launch_quantize_rows_fp8(const __nv_bfloat16* a, const int32_t* src, int R, int C, int src_rows,
                                     uint8_t* q, float* scale, int32_t* status, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    return launch_k(kPdlQuant, quantize_rows_kernel, dim3(R), dim3(kQThreads), 0, s,
                    reinterpret_cast<const uint4*>(a), src, R, C, src_rows, reinterpret_cast<uint2*>(q), scale,
                    status);
}

cudaError_t launch_quantize_weights_fp8(const __nv_bfloat16* W, int E, int K, int N, uint8_t* Wq, float* scale,
                                        cudaStream_t s) {
    if (reinterpret_cast<uintptr_t>(W) & 15u) {  // 16-byte loads need an aligned W: the two-pass kernel
        const dim3 grid((N + kWCols - 1) / kWCols, E);
        quantize_weights_kernel<<<grid, kQThreads, 0, s>>>(reinterpret_cast<const uint16_t*>(W), K, N, Wq, scale);
        return cudaGetLastError();
    }
    // scale holds the column maxima (as bits) until the last step turns them into scales.
    cudaError_t e = cudaMemsetAsync(scale, 0, static_cast<size_t>(E) * N * sizeof(float), s);
    if (e != cudaSuccess) return e;
    const uint4* W4 = reinterpret_cast<const uint4*>(W);
    weights_colmax_kernel<<<dim3((N + kCmCols - 1) / kCmCols, (K + kCmRows - 1) / kCmRows, E), kQThreads, 0, s>>>(
        W4, K, N, reinterpret_cast<unsigned int*>(scale));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    weights_tile_kernel<<<dim3(N / 64, K / 128, E), kQThreads, 0, s>>>(W4, K, N, scale, Wq);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int n = E * N;
    colmax_to_scale_kernel<<<(n + kQThreads - 1) / kQThreads, kQThreads, 0, s>>>(scale, n);
    return cudaGetLastError();
}

}  // namespace moe
