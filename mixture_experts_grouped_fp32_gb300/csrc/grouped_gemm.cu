// grouped_gemm.cu — steps 3 and 4: the two grouped BF16 GEMMs of the MoE layer on the sm_103a
// tensor cores (TMA -> shared memory -> tcgen05.mma -> tensor memory -> epilogue).
//
//   kind 0, gate+up+SwiGLU: for the rows r of expert e, [g | u] = x_perm[r] . W_gate_up[e]
//           (K = d), h[r] = bf16(silu(g) * u).  The fp32 g and u exist only in tensor memory —
//           the gate/up fusion that keeps the SwiGLU intermediate out of global memory
//           ("Triton-MoE-Dispatch-Kernel erreicht 131 % von Megablocks", lumeric.app).
//   kind 1, down: y_perm[r] = h[r] . W_down[e] (K = f), fp32 out.
//
// Work decomposition ("block-scheduled grouped GEMM for variable expert batches":
// "Triton MoE 核心擊敗 Megablocks", setupai.cc, section 關鍵要點).  Expert e's rows form
// ceil(count_e / 128) M-tiles; each (expert, N-tile, M-tile) is one work item of identical cost
// (same K, full 128x256 MMA tile), so a static round-robin over a persistent grid of one CTA per
// SM balances any expert skew up to one item.  Items are numbered expert-major, then N-tile,
// then M-tile, so CTAs that run together share a weight tile (in L2) and an expert's activation
// rows stay L2-resident while its N-tiles sweep ("persistent cache-aware" strategy:
// "Triton-Optimierter BF16 Grouped GEMM Kernel beschleunigt MoE-Modelle", meineki.news).  The
// persistent kernel overlaps one tile's epilogue with the next tile's main loop through two
// tensor-memory accumulators (HPC-Ops page: persistent kernels hide prologue/epilogue cost).
//
// Roles (warp specialisation as in the DeepGEMM write-up, section 1.2, technique 2, without the
// communication role): warp 0 lane 0 issues TMA loads into a 4-stage ring; warp 1 owns tensor
// memory and lane 0 issues tcgen05.mma; warps 2-5 (128 threads, one accumulator row each) run
// the epilogue.  Every wait is bounded (1 s) and reports MOE_STATUS_WAIT_TIMEOUT instead of
// hanging.
//
// Shared-memory operand layouts (128-byte swizzle, as written by TMA with SWIZZLE_128B):
//   A (activations, K-major): 128 rows x 64 K, row pitch 128 B, 8-row groups 1024 B apart.
//   B (weights [K, N] with N contiguous, i.e. MN-major): four 64-column boxes of 64 K-rows,
//     8 KB apart; inside a box, K-row pitch 128 B, 8-row groups 1024 B apart.
//   UMMA: M = 128, N = 256, K = 16 per instruction, fp32 accumulator = 256 TMEM columns.
#include "common.cuh"
#include "tcgen05.cuh"

#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

namespace moe {
namespace {

constexpr int BM = 128;                         // tile rows = UMMA M
constexpr int BK = 64;                          // K per stage (one 128-byte swizzle row)
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BOX_N = 64;
constexpr int B_BOXES = 4;
constexpr int B_BOX_BYTES = B_BOX_N * BK * 2;   // 8 KB
constexpr int B_BYTES = B_BOXES * B_BOX_BYTES;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int UMMA_N = B_BOXES * B_BOX_N;       // 256
constexpr int ACC_COLS = UMMA_N;                // fp32 columns per accumulator
constexpr int NUM_ACC = 2;
constexpr int TMEM_COLS = NUM_ACC * ACC_COLS;   // 512
constexpr int NUM_THREADS = 192;
constexpr int MAX_E = 256;
// The whole opt-in shared memory of an SM: one CTA per SM, and any descriptor mistake would
// still read inside this CTA's own allocation.
constexpr int SMEM_BYTES = 232448;

struct Ctl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[NUM_ACC];
    uint64_t tempty[NUM_ACC];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int total_items;
    int seg[MAX_E + 1];         // copy of offsets[]
    int item_start[MAX_E + 1];  // first work item of each expert
};
static_assert(STAGES * STAGE_BYTES + 1024 + sizeof(Ctl) <= SMEM_BYTES, "shared memory budget");

struct Item {
    int e, n_tile, m_tile, row0, rows;
};

__device__ __forceinline__ Item decode_item(const Ctl& c, int E, int i) {
    int lo = 0, hi = E;  // item_start[lo] <= i < item_start[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (c.item_start[mid] <= i) lo = mid; else hi = mid;
    }
    Item it;
    it.e = lo;
    const int cnt = c.seg[lo + 1] - c.seg[lo];
    const int mt = (cnt + BM - 1) / BM;
    const int j = i - c.item_start[lo];
    it.n_tile = j / mt;
    it.m_tile = j - it.n_tile * mt;
    it.row0 = c.seg[lo] + it.m_tile * BM;
    it.rows = min(BM, cnt - it.m_tile * BM);
    return it;
}

__device__ __forceinline__ void raise_abort(Ctl& c, int32_t* status) {
    *reinterpret_cast<volatile int*>(&c.abort_flag) = 1;
    flag_status(status, MOE_STATUS_WAIT_TIMEOUT);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return g / (1.0f + __expf(-g)) * u;
}

// KIND 0: gate+up+SwiGLU (output tile = 128 h columns, B boxes = gate n0, n0+64, up f+n0, f+n0+64)
// KIND 1: down             (output tile = 256 y columns, B boxes = n0 + 64 q)
template <int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const int32_t* __restrict__ offsets, int M, int K, int N, int E,
                    void* __restrict__ out, int32_t* __restrict__ status) {
    constexpr int BN_OUT = KIND == 0 ? 128 : 256;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    uint8_t* tiles = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    Ctl& c = *reinterpret_cast<Ctl*>(tiles + STAGES * STAGE_BYTES);
    const volatile int* abort_flag = &c.abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_tiles = (N + BN_OUT - 1) / BN_OUT;
    const int num_kb = K / BK;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&c.full[s], 1);
            ptx::mbar_init(&c.empty[s], 1);
        }
        for (int a = 0; a < NUM_ACC; ++a) {
            ptx::mbar_init(&c.tfull[a], 1);
            ptx::mbar_init(&c.tempty[a], 4);
        }
        ptx::mbar_init(&c.drain, 1);
        c.abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&c.tmem_base, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == 2) {
        // Validate offsets and build the per-expert item prefix (8 experts per lane).
        for (int e = lane; e <= E; e += 32) c.seg[e] = __ldg(offsets + e);
        __syncwarp();
        bool ok = true;
        for (int e = lane; e < E; e += 32) ok = ok && c.seg[e] <= c.seg[e + 1];
        if (lane == 0) ok = ok && c.seg[0] >= 0 && c.seg[E] <= M;
        ok = __all_sync(0xffffffffu, ok);
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        int sum = 0;
        if (ok)
            for (int e = e0; e < e1; ++e) sum += ((c.seg[e + 1] - c.seg[e] + BM - 1) / BM) * n_tiles;
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int e = e0; e < e1; ++e) {
            c.item_start[e] = run;
            if (ok) run += ((c.seg[e + 1] - c.seg[e] + BM - 1) / BM) * n_tiles;
        }
        if (lane == 31) {
            c.item_start[E] = incl;
            c.total_items = incl;
        }
        if (!ok && lane == 0) flag_status(status, MOE_STATUS_BAD_OFFSETS);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    const uint32_t tmem_base = c.tmem_base;
    const int total = c.total_items;
    uint32_t fill_parity[STAGES];  // producer: parity of each stage's most recent fill
    int filled_mask = 0;

    if (warp == 0 && lane == 0) {
        // ------------------------------ TMA producer ------------------------------
        const uint64_t pol_act = ptx::policy_evict_last();   // activations: reused across N-tiles
        const uint64_t pol_wgt = ptx::policy_evict_normal();  // weights: shared by an item's M-tiles
        uint32_t stage = 0, phase = 0;
        bool aborted = false;
        for (int i = blockIdx.x; i < total && !aborted; i += gridDim.x) {
            const Item it = decode_item(c, E, i);
            const int n0 = it.n_tile * BN_OUT;
            const int brow = it.e * K;
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!ptx::mbar_wait(&c.empty[stage], phase ^ 1u, abort_flag)) {
                    raise_abort(c, status);
                    aborted = true;
                    break;
                }
                uint8_t* sa = tiles + stage * STAGE_BYTES;
                uint8_t* sb = sa + A_BYTES;
                ptx::mbar_arrive_expect_tx(&c.full[stage], STAGE_BYTES);
                ptx::tma_load_2d(sa, &tmA, &c.full[stage], kb * BK, it.row0, pol_act);
#pragma unroll
                for (int q = 0; q < B_BOXES; ++q) {
                    int col;
                    if (KIND == 0) col = (q < 2) ? n0 + q * B_BOX_N : N + n0 + (q - 2) * B_BOX_N;
                    else col = n0 + q * B_BOX_N;
                    ptx::tma_load_2d(sb + q * B_BOX_BYTES, &tmB, &c.full[stage], col, brow + kb * BK,
                                     pol_wgt);
                }
                fill_parity[stage] = phase;
                filled_mask |= 1 << stage;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------ MMA issuer ------------------------------
        constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, UMMA_N, /*a_mn=*/0, /*b_mn=*/1);
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool aborted = false;
        for (int i = blockIdx.x; i < total && !aborted; i += gridDim.x) {
            if (!ptx::mbar_wait(&c.tempty[acc], acc_phase ^ 1u, abort_flag)) {
                raise_abort(c, status);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!ptx::mbar_wait(&c.full[stage], phase, abort_flag)) {
                    raise_abort(c, status);
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sa = ptx::smem_u32(tiles + stage * STAGE_BYTES);
                const uint64_t a_desc = ptx::smem_desc_sw128(sa, 16, 1024);
                const uint64_t b_desc = ptx::smem_desc_sw128(sa + A_BYTES, B_BOX_BYTES, 1024);
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                    // K-major A: +32 bytes per 16 K; MN-major B: +16 rows * 128 bytes per 16 K.
                    ptx::mma_bf16_ss(d_tmem, a_desc + static_cast<uint64_t>((kk * 32) >> 4),
                                     b_desc + static_cast<uint64_t>((kk * 2048) >> 4), idesc,
                                     (kb | kk) != 0 ? 1u : 0u);
                }
                ptx::mma_commit(&c.empty[stage]);  // frees the stage once these MMAs finish
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (aborted) break;
            ptx::mma_commit(&c.tfull[acc]);  // accumulator ready for the epilogue
            if (++acc == NUM_ACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    } else if (warp >= 2) {
        // ------------------------------ epilogue ------------------------------
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 belong to this warp
        const int r_local = quarter * 32 + lane;
        uint32_t acc = 0, acc_phase = 0;
        for (int i = blockIdx.x; i < total; i += gridDim.x) {
            const Item it = decode_item(c, E, i);
            if (!ptx::mbar_wait(&c.tfull[acc], acc_phase, abort_flag)) {
                raise_abort(c, status);
                break;
            }
            ptx::tc_fence_after();
            const bool row_ok = r_local < it.rows;
            const size_t grow = static_cast<size_t>(it.row0 + r_local);
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * ACC_COLS;
            const int n0 = it.n_tile * BN_OUT;
            if (KIND == 0) {
                __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(out);
#pragma unroll 1
                for (int cc = 0; cc < BN_OUT / 32; ++cc) {
                    uint32_t g[32], u[32];
                    ptx::tmem_ld_32x32b_x32(taddr + cc * 32, g);
                    ptx::tmem_ld_32x32b_x32(taddr + 128 + cc * 32, u);
                    ptx::tmem_ld_wait();
                    const int col = n0 + cc * 32;
                    if (row_ok && col < N) {
                        uint4* dst = reinterpret_cast<uint4*>(h + grow * N + col);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 o;
                            o.x = pack_bf16x2(silu_mul(__uint_as_float(g[8 * v + 0]), __uint_as_float(u[8 * v + 0])),
                                              silu_mul(__uint_as_float(g[8 * v + 1]), __uint_as_float(u[8 * v + 1])));
                            o.y = pack_bf16x2(silu_mul(__uint_as_float(g[8 * v + 2]), __uint_as_float(u[8 * v + 2])),
                                              silu_mul(__uint_as_float(g[8 * v + 3]), __uint_as_float(u[8 * v + 3])));
                            o.z = pack_bf16x2(silu_mul(__uint_as_float(g[8 * v + 4]), __uint_as_float(u[8 * v + 4])),
                                              silu_mul(__uint_as_float(g[8 * v + 5]), __uint_as_float(u[8 * v + 5])));
                            o.w = pack_bf16x2(silu_mul(__uint_as_float(g[8 * v + 6]), __uint_as_float(u[8 * v + 6])),
                                              silu_mul(__uint_as_float(g[8 * v + 7]), __uint_as_float(u[8 * v + 7])));
                            dst[v] = o;
                        }
                    }
                }
            } else {
                float* y = reinterpret_cast<float*>(out);
#pragma unroll 1
                for (int cc = 0; cc < BN_OUT / 32; ++cc) {
                    uint32_t v32[32];
                    ptx::tmem_ld_32x32b_x32(taddr + cc * 32, v32);
                    ptx::tmem_ld_wait();
                    const int col = n0 + cc * 32;
                    if (row_ok && col < N) {
                        float4* dst = reinterpret_cast<float4*>(y + grow * N + col);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            dst[v] = make_float4(__uint_as_float(v32[4 * v]), __uint_as_float(v32[4 * v + 1]),
                                                 __uint_as_float(v32[4 * v + 2]), __uint_as_float(v32[4 * v + 3]));
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&c.tempty[acc]);
            if (++acc == NUM_ACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    // ------------------------------ teardown ------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0 && c.abort_flag) {
        // Let this CTA's own TMA copies land before its shared memory is released.
        for (int s = 0; s < STAGES; ++s)
            if (filled_mask & (1 << s)) ptx::mbar_wait_ns(&c.full[s], fill_parity[s], 100000000ull);
    }
    if (warp == 1 && lane == 0) {
        // Every MMA this thread issued has completed once this commit arrives.
        ptx::mma_commit(&c.drain);
        ptx::mbar_wait_ns(&c.drain, 0, 100000000ull);
    }
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), box = [box_rows, 64 cols], 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND>
cudaError_t launch_kind(const GemmArgs& a, int num_sms, cudaStream_t s, const char** why) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<KIND>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) {
            *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
            return e;
        }
        attr_set[dev] = true;
    }
    CUtensorMap mA, mB;
    const uint64_t bcols = KIND == 0 ? 2ull * a.N : static_cast<uint64_t>(a.N);
    if (!make_map(&mA, a.A, a.K, a.M, BM) ||
        !make_map(&mB, a.B, bcols, static_cast<uint64_t>(a.E) * a.K, BK)) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point missing or bad operand)";
        return cudaErrorInvalidValue;
    }
    grouped_gemm_kernel<KIND><<<num_sms, NUM_THREADS, SMEM_BYTES, s>>>(
        mA, mB, a.offsets, a.M, a.K, a.N, a.E, a.out, a.status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm(int kind, const GemmArgs& a, int num_sms, cudaStream_t s,
                                const char** why) {
    return kind == 0 ? launch_kind<0>(a, num_sms, s, why) : launch_kind<1>(a, num_sms, s, why);
}

}  // namespace moe
