// grouped_gemm_2sm.cu — the two grouped GEMMs of the MoE layer on pairs of SMs (tcgen05
// cta_group::2), for launches whose experts hold 128 rows or more on average.
//
// Same operation and item order as grouped_gemm.cu (normal orientation only), but each work
// item is a 256-row tile computed by a cluster of two CTAs on two SMs:
//   * CTA r of the pair owns activation rows row0 + 128 r .. +127 (its M-tile) and loads them;
//   * the 256 weight columns of the tile are split: each CTA loads its 128-column half;
//   * one thread of CTA 0 issues M=256 x N=256 UMMAs that read both CTAs' shared memory and
//     accumulate CTA r's 128 rows into CTA r's tensor memory.
// Per 64-deep K block each SM thus fills 32 KB of shared memory (16 KB rows + 16 KB half weights)
// instead of 48 KB, and the weight tile is fetched once for both M-tiles.  Sibling M-tiles of an
// expert share one weight load instead of two.
//
// Synchronisation across the pair:
//   full[s]   lives in CTA 0: its producer arms it with the bytes of both CTAs; both producers'
//             TMA loads complete on it (cp.async.bulk.tensor .cta_group::2).
//   empty[s]  in each CTA: CTA 0's MMA commit multicasts one arrive to both.
//   tfull[a]  in each CTA: CTA 0's commit multicasts when accumulator a is final.
//   tempty[a] lives in CTA 0: all 8 epilogue warps of the pair arrive (peer warps remotely).
// Every wait is bounded as in grouped_gemm.cu.
#include "common.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace {

constexpr int BM = 128;          // rows per CTA (M-tile)
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;         // 8 KB
constexpr int BH_BOXES = 2;                      // weight boxes per CTA (half of the tile)
constexpr int BH_BYTES = BH_BOXES * B_BOX_BYTES; // 16 KB
constexpr int STAGE_BYTES = A_BYTES + BH_BYTES;  // 32 KB
constexpr int PAIR_STAGE_BYTES = 2 * STAGE_BYTES;
constexpr int ACC_COLS = 256;
constexpr int NUM_ACC = 2;
constexpr int TMEM_COLS = NUM_ACC * ACC_COLS;
constexpr int NUM_THREADS = 192;
constexpr int MAX_E = 256;
constexpr int SMEM_BYTES = 232448;
constexpr uint16_t BOTH_CTAS = 0x3;

struct Ctl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[NUM_ACC];
    uint64_t tempty[NUM_ACC];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int total_items;
    int seg[MAX_E + 1];
    int item_start[MAX_E + 1];
};
static_assert(STAGES * STAGE_BYTES + 1024 + sizeof(Ctl) <= SMEM_BYTES, "shared memory budget");

struct PairItem {
    int e, n_tile, kslice, row0, rows;  // row0/rows: this CTA's M-tile (rows may be <= 0)
};

// Items of expert e: ceil(ceil(count / 128) / 2) M-tile pairs x n_tiles x ksplit, ordered N-tile,
// pair, K-slice.
__device__ __forceinline__ PairItem decode_pair_item(const Ctl& c, int E, int ksplit, int rank, int i) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (c.item_start[mid] <= i) lo = mid; else hi = mid;
    }
    PairItem it;
    it.e = lo;
    const int cnt = c.seg[lo + 1] - c.seg[lo];
    const int pairs = ((cnt + BM - 1) / BM + 1) / 2;
    const int j = i - c.item_start[lo];
    const int per_n = pairs * ksplit;
    it.n_tile = j / per_n;
    const int r = j - it.n_tile * per_n;
    const int mpair = r / ksplit;
    it.kslice = r - mpair * ksplit;
    const int mtile = 2 * mpair + rank;
    it.row0 = c.seg[lo] + mtile * BM;
    it.rows = min(BM, cnt - mtile * BM);
    return it;
}

__device__ __forceinline__ void raise_abort(Ctl& c, int32_t* status) {
    *reinterpret_cast<volatile int*>(&c.abort_flag) = 1;
    flag_status(status, MOE_STATUS_WAIT_TIMEOUT);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return g / (1.0f + __expf(-g)) * u;
}

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const int32_t* __restrict__ offsets, int M, int K, int N, int E, int ksplit,
                        void* __restrict__ out, int32_t* __restrict__ status) {
    constexpr int BN_OUT = KIND == 0 ? 128 : 256;  // output columns of a tile
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    uint8_t* tiles = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    Ctl& c = *reinterpret_cast<Ctl*>(tiles + STAGES * STAGE_BYTES);
    const volatile int* abort_flag = &c.abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = static_cast<int>(ptx::cluster_ctarank());
    const bool leader = rank == 0;
    const int pair_id = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
    const int n_tiles = (N + BN_OUT - 1) / BN_OUT;
    const int num_kb = K / BK;
    const int kb_per = (num_kb + ksplit - 1) / ksplit;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&c.full[s], 1);
            ptx::mbar_init(&c.empty[s], 1);
        }
        for (int a = 0; a < NUM_ACC; ++a) {
            ptx::mbar_init(&c.tfull[a], 1);
            ptx::mbar_init(&c.tempty[a], 8);
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
        ptx::tmem_alloc_pair(&c.tmem_base, TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    pdl_wait();
    pdl_trigger();
    if (warp == 2) {
        for (int e = lane; e <= E; e += 32) c.seg[e] = __ldg(offsets + e);
        __syncwarp();
        bool ok = true;
        for (int e = lane; e < E; e += 32) ok = ok && c.seg[e] <= c.seg[e + 1];
        if (lane == 0) ok = ok && c.seg[0] >= 0 && c.seg[E] <= M;
        ok = __all_sync(0xffffffffu, ok);
        const int per = (E + 31) / 32;
        const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
        const int per_tile = n_tiles * ksplit;
        int sum = 0;
        if (ok)
            for (int e = e0; e < e1; ++e) sum += (((c.seg[e + 1] - c.seg[e] + BM - 1) / BM + 1) / 2) * per_tile;
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int e = e0; e < e1; ++e) {
            c.item_start[e] = run;
            if (ok) run += (((c.seg[e + 1] - c.seg[e] + BM - 1) / BM + 1) / 2) * per_tile;
        }
        if (lane == 31) {
            c.item_start[E] = incl;
            c.total_items = incl;
        }
        if (!ok && lane == 0 && leader) flag_status(status, MOE_STATUS_BAD_OFFSETS);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrive or copy
    ptx::tc_fence_after();

    const uint32_t tmem_base = c.tmem_base;
    const int total = c.total_items;
    uint32_t fill_parity[STAGES];
    int filled_mask = 0;

    if (warp == 0 && lane == 0) {
        // ------------------------------ TMA producer (both CTAs) ------------------------------
        const uint64_t pol_act = ptx::policy_evict_last();
        const uint64_t pol_wgt = ptx::policy_evict_normal();
        uint32_t stage = 0, phase = 0;
        bool aborted = false;
        for (int i = pair_id; i < total && !aborted; i += num_pairs) {
            const PairItem it = decode_pair_item(c, E, ksplit, rank, i);
            const int n0 = it.n_tile * BN_OUT;
            const int brow = it.e * K;
            const int kb0 = it.kslice * kb_per, kb1 = min(num_kb, kb0 + kb_per);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!ptx::mbar_wait(&c.empty[stage], phase ^ 1u, abort_flag)) {
                    raise_abort(c, status);
                    aborted = true;
                    break;
                }
                uint8_t* sa = tiles + stage * STAGE_BYTES;
                uint8_t* sb = sa + A_BYTES;
                const uint32_t full_leader = ptx::map_to_cta(ptx::smem_u32(&c.full[stage]), 0);
                if (leader) ptx::mbar_arrive_expect_tx(&c.full[stage], PAIR_STAGE_BYTES);
                ptx::tma_load_2d_pair(sa, &tmA, full_leader, kb * BK, it.row0, pol_act);
#pragma unroll
                for (int q = 0; q < BH_BOXES; ++q) {
                    // kind 0: CTA r holds gate columns n0+64r.. and up columns f+n0+64r..;
                    // kind 1: CTA r holds output columns n0+128r .. n0+128r+127.
                    const int col = KIND == 0 ? (q == 0 ? n0 + 64 * rank : N + n0 + 64 * rank)
                                              : n0 + 128 * rank + 64 * q;
                    ptx::tma_load_2d_pair(sb + q * B_BOX_BYTES, &tmB, full_leader, col, brow + kb * BK, pol_wgt);
                }
                fill_parity[stage] = phase;
                filled_mask |= 1 << stage;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------ pair MMA issuer (CTA 0) ------------------------------
        constexpr uint32_t idesc = ptx::idesc_bf16_f32(2 * BM, ACC_COLS, /*a_mn=*/0, /*b_mn=*/1);
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool aborted = false;
        for (int i = pair_id; i < total && !aborted; i += num_pairs) {
            const PairItem it = decode_pair_item(c, E, ksplit, rank, i);
            const int kb0 = it.kslice * kb_per, kb1 = min(num_kb, kb0 + kb_per);
            if (!ptx::mbar_wait(&c.tempty[acc], acc_phase ^ 1u, abort_flag)) {
                raise_abort(c, status);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
            for (int kb = kb0; kb < kb1; ++kb) {
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
                for (int kk = 0; kk < BK / UMMA_K; ++kk)
                    ptx::mma_bf16_ss_pair(d_tmem, a_desc + static_cast<uint64_t>((kk * 32) >> 4),
                                          b_desc + static_cast<uint64_t>((kk * 2048) >> 4), idesc,
                                          (kb != kb0 || kk != 0) ? 1u : 0u);
                ptx::mma_commit_pair(&c.empty[stage], BOTH_CTAS);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (aborted) break;
            ptx::mma_commit_pair(&c.tfull[acc], BOTH_CTAS);
            if (++acc == NUM_ACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    } else if (warp >= 2) {
        // ------------------------------ epilogue (both CTAs) ------------------------------
        const int quarter = warp & 3;
        const int r_local = quarter * 32 + lane;
        uint32_t acc = 0, acc_phase = 0;
        for (int i = pair_id; i < total; i += num_pairs) {
            const PairItem it = decode_pair_item(c, E, ksplit, rank, i);
            if (!ptx::mbar_wait(&c.tfull[acc], acc_phase, abort_flag)) {
                raise_abort(c, status);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * ACC_COLS;
            const int n0 = it.n_tile * BN_OUT;
            const bool kfull = it.kslice * kb_per < num_kb;  // an empty K slice contributes zeros
            const bool row_ok = r_local < it.rows;
            const size_t grow = static_cast<size_t>(it.row0 + r_local);
            if (KIND == 0) {
                // Accumulator columns: [gate n0..+63 | up n0..+63 | gate n0+64..+127 | up n0+64..+127].
                __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(out);
#pragma unroll 1
                for (int cc = 0; cc < BN_OUT / 32; ++cc) {
                    const uint32_t gcol = (cc < 2 ? 32 * cc : 128 + 32 * (cc - 2));
                    uint32_t g[32], u[32];
                    ptx::tmem_ld_32x32b_x32(taddr + gcol, g);
                    ptx::tmem_ld_32x32b_x32(taddr + gcol + 64, u);
                    ptx::tmem_ld_wait();
                    const int col = n0 + cc * 32;
                    if (row_ok && col < N) {
                        uint4* dst = reinterpret_cast<uint4*>(h + grow * N + col);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint32_t p[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                p[q] = pack_bf16x2(
                                    silu_mul(__uint_as_float(g[8 * v + 2 * q]), __uint_as_float(u[8 * v + 2 * q])),
                                    silu_mul(__uint_as_float(g[8 * v + 2 * q + 1]), __uint_as_float(u[8 * v + 2 * q + 1])));
                            dst[v] = make_uint4(p[0], p[1], p[2], p[3]);
                        }
                    }
                }
            } else {
                float* y = reinterpret_cast<float*>(out) + static_cast<size_t>(it.kslice) * M * N;
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
                            dst[v] = make_float4(kfull ? __uint_as_float(v32[4 * v]) : 0.0f,
                                                 kfull ? __uint_as_float(v32[4 * v + 1]) : 0.0f,
                                                 kfull ? __uint_as_float(v32[4 * v + 2]) : 0.0f,
                                                 kfull ? __uint_as_float(v32[4 * v + 3]) : 0.0f);
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(ptx::map_to_cta(ptx::smem_u32(&c.tempty[acc]), 0));
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
        if (leader) {
            // CTA 0's full barriers count both CTAs' copies: wait for every stage filled so far.
            for (int s = 0; s < STAGES; ++s)
                if (filled_mask & (1 << s)) ptx::mbar_wait_ns(&c.full[s], fill_parity[s], 100000000ull);
        } else {
            const uint64_t t0 = ptx::globaltimer_ns();  // give this CTA's own copies time to land
            while (ptx::globaltimer_ns() - t0 < 1000000ull) {
            }
        }
    }
    if (warp == 1 && lane == 0 && leader) {
        ptx::mma_commit_pair(&c.drain, 0x1);  // all pair MMAs issued by this thread have completed
        ptx::mbar_wait_ns(&c.drain, 0, 100000000ull);
    }
    __syncthreads();
    ptx::cluster_sync();  // neither CTA frees tensor memory or exits while the pair MMAs may run
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    ptx::cluster_sync();
}

template <int KIND>
cudaError_t launch_pair_kind(const GemmArgs& a, int num_sms, cudaStream_t s, const char** why) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_2sm_kernel<KIND>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) {
            *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
            return e;
        }
        attr_set[dev] = true;
    }
    CUtensorMap mA, mB;
    const uint64_t bcols = KIND == 0 ? 2ull * a.N : static_cast<uint64_t>(a.N);
    if (!make_tensor_map_bf16(&mA, a.A, a.K, a.M, BM) ||
        !make_tensor_map_bf16(&mB, a.B, bcols, static_cast<uint64_t>(a.E) * a.K, BK)) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point missing or bad operand)";
        return cudaErrorInvalidValue;
    }
    const int grid = num_sms & ~1;  // whole CTA pairs
    const int ksplit = KIND == 0 ? 1 : a.ksplit;
    return launch_k(KIND == 0 ? kPdlGateUp : kPdlDown, grouped_gemm_2sm_kernel<KIND>, dim3(grid),
                    dim3(NUM_THREADS), SMEM_BYTES, s, mA, mB, a.offsets, a.M, a.K, a.N, a.E, ksplit, a.out,
                    a.status);
}

}  // namespace

cudaError_t launch_grouped_gemm_pair(int kind, const GemmArgs& a, int num_sms, cudaStream_t s,
                                     const char** why) {
    return kind == 0 ? launch_pair_kind<0>(a, num_sms, s, why) : launch_pair_kind<1>(a, num_sms, s, why);
}

}  // namespace moe
