// grouped_gemm.cu — steps 3 and 4: the two grouped BF16 GEMMs of the MoE layer on the sm_103a
// tensor cores (TMA -> shared memory -> tcgen05.mma -> tensor memory -> epilogue).
//
//   kind 0, gate+up+SwiGLU: for the rows r of expert e, [g | u] = x_perm[r] . W_gate_up[e]
//           (K = d), h[r] = bf16(silu(g) * u).  The fp32 g and u exist only in tensor memory —
//           the gate/up fusion that keeps the SwiGLU intermediate out of global memory
//           ("Triton-MoE-Dispatch-Kernel erreicht 131 % von Megablocks", lumeric.app).
//   kind 1, down: y_perm[r] = h[r] . W_down[e] (K = f), fp32 out, optionally split over K into
//           `ksplit` partial slices that the combine step adds in a fixed order.
//
// Work decomposition ("block-scheduled grouped GEMM for variable expert batches":
// "Triton MoE 核心擊敗 Megablocks", setupai.cc, section 關鍵要點).  Expert e's rows form
// ceil(count_e / 128) M-tiles; each (expert, N-tile, M-tile, K-slice) is one work item, and items
// of one launch all cost the same weight bytes, so a static round-robin over a persistent grid of
// one CTA per SM balances any expert skew to within one item.  Items are numbered expert-major,
// then N-tile, M-tile, K-slice, so CTAs that run together share a weight tile (in L2) and an
// expert's activation rows stay L2-resident while its N-tiles sweep ("persistent cache-aware"
// strategy: "Triton-Optimierter BF16 Grouped GEMM Kernel beschleunigt MoE-Modelle",
// meineki.news).  Two tensor-memory accumulators let one item's epilogue overlap the next item's
// main loop (HPC-Ops page: persistent kernels hide prologue/epilogue cost).
//
// Two operand orientations, chosen per item from the expert's row count on the device:
//   normal   UMMA M = 128 activation rows, N = 256 weight columns (the expert has > swap_max rows)
//   swap-AB  UMMA M = 128 weight columns, N = the expert's rows rounded up to 16 (<= swap_max):
//            the weights become the A operand so a small expert costs an N=16..128 MMA instead
//            of a mostly empty 128-row tile, and only ceil(rows/32) 32-row activation boxes are
//            loaded (DeepGEMM write-up, section 3.2, "dynamic swap A/B": B^T . A^T puts the large,
//            regular weight dimension on the UMMA M side).
//
// Roles (warp specialisation as in the DeepGEMM write-up, section 1.2, technique 2, without the
// communication role): warp 0 lane 0 issues TMA loads into a 4-stage ring; warp 1 owns tensor
// memory and lane 0 issues tcgen05.mma; warps 2-5 (128 threads, one accumulator lane each) run
// the epilogue.  Every wait is bounded (1 s) and reports MOE_STATUS_WAIT_TIMEOUT instead of
// hanging.
//
// Shared-memory stage (128-byte swizzle, as written by TMA with SWIZZLE_128B), 48 KB:
//   activations, K-major: up to 128 rows x 64 K, row pitch 128 B, 8-row groups 1024 B apart.
//   weights ([K, N] with N contiguous, i.e. MN-major): four 64-column boxes of 64 K-rows, 8 KB
//     apart; inside a box, K-row pitch 128 B, 8-row groups 1024 B apart.  For kind 0 the boxes
//     hold gate columns n0..n0+127 then up columns f+n0..f+n0+127.
//   normal mode: one M=128 x N=256 MMA per 16-deep K step into a 256-column fp32 accumulator
//     (kind 0: columns 0-127 gate, 128-255 up).
//   swap mode: two M=128 x N=rows16 MMAs per K step, weight boxes 0-1 and 2-3 as A, into
//     accumulator columns [0, N) and [128, 128+N) (kind 0: gate and up; kind 1: output columns
//     n0..n0+127 and n0+128..n0+255).
//
// FP8 variant (E4M3 codes, kind::f8f6f4 MMAs with K = 32): the activations are [M, K] codes with a
// scale per row, the weights are stored transposed and blocked, [E * N_total / 64, K / 128, 64, 128]
// codes (64 output columns x 128 K values per contiguous 8 KB block) with a scale per output
// column, so both operands are K-major and one 128-byte swizzle row holds 128 K values: a stage is
// 128 K deep, and each weight box is one or two whole 8 KB blocks of HBM rather than 128 rows of
// 128 bytes a power-of-two stride apart.  (Row-major [N, K] codes with K = 4096 streamed ~10 %
// slower even in the pure weight-streaming case, and up to ~25 % slower at 128-256 rows per
// expert.)  Its weight part is two 128-row boxes (kind 0: gate rows n0.. and
// up rows f+n0..; kind 1: rows n0.. and n0+128..), 16 KB each, and the accumulator columns keep the
// BF16 kernel's meaning.  The scales factor out of the K sum, so the epilogue multiplies each
// accumulator by scale_row * scale_col before SwiGLU (kind 0) or the store (kind 1).
#include "common.cuh"
#include "tcgen05.cuh"

#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

namespace moe {
namespace {

constexpr int BM = 128;                         // activation rows per M-tile
constexpr int BK = 64;                          // K per stage (one 128-byte swizzle row)
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int A_BOX32_ROWS = 32;                // activation box height in swap mode
constexpr int A_BOX32_BYTES = A_BOX32_ROWS * BK * 2;  // 4 KB
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
// GATHER launches add kGatherWarps warps (6..9) that gather the activation rows, one per ring
// slot: a warp then never waits on a slot's `empty` barrier more than one phase ahead (which its
// parity wait requires).
constexpr int kGatherWarps = STAGES;
constexpr int kGatherWarp0 = NUM_THREADS / 32;
constexpr int GATHER_THREADS = NUM_THREADS + 32 * kGatherWarps;
constexpr int MAX_E = 256;
constexpr int SWAP_MAX_ROWS = 128;              // swap mode needs N = rows16 <= 128
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
    int e, n_tile, m_tile, kslice, row0, rows;
    bool swap;
};

// Items of expert e: ceil(count / BM) M-tiles x n_tiles x ksplit, ordered N-tile, M-tile, K-slice.
__device__ __forceinline__ Item decode_item(const Ctl& c, int E, int ksplit, int swap_max, int i) {
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
    const int per_n = mt * ksplit;
    it.n_tile = j / per_n;
    const int r = j - it.n_tile * per_n;
    it.m_tile = r / ksplit;
    it.kslice = r - it.m_tile * ksplit;
    it.row0 = c.seg[lo] + it.m_tile * BM;
    it.rows = min(BM, cnt - it.m_tile * BM);
    it.swap = cnt <= swap_max;
    return it;
}

__device__ __forceinline__ void raise_abort(Ctl& c, int32_t* status) {
    *reinterpret_cast<volatile int*>(&c.abort_flag) = 1;
    flag_status(status, MOE_STATUS_WAIT_TIMEOUT);
}

// silu(g) * u = g / (1 + e^-g) * u, with CUDA's fast-divide intrinsic: its error (~2 ulp) is far
// below the bf16 rounding of h that follows (for g below about -88, 1 + e^-g is infinite and the
// quotient is -0, as silu's limit).
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__device__ __forceinline__ uint16_t bf16_bits(float v) {
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&b);
}

// KIND 0: gate+up+SwiGLU (output tile = 128 h columns; weight boxes gate n0, n0+64, up f+n0, f+n0+64)
// KIND 1: down             (output tile = 256 y columns; weight boxes n0 + 64 q)
// GATHER (kind 0 only): the activation rows are not read from x_perm with TMA but gathered from x
// by the permutation's src[] with 16-byte cp.async copies, issued by four extra warps into the
// 128-byte-swizzled positions TMA would have written; rows past the expert's end are zero-filled.
// Each stage's `full` barrier then expects two arrivals: the TMA weight bytes' and its gather
// warp's.  x_perm then never exists in global memory.
template <int KIND, bool GATHER, bool FP8>
__global__ void __launch_bounds__(GATHER ? GATHER_THREADS : NUM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA32,
                    const __grid_constant__ CUtensorMap tmB, const int32_t* __restrict__ offsets, int M,
                    int K, int N, int E, int ksplit, int swap_max, int inject_stall,
                    const int4* __restrict__ xg, const int32_t* __restrict__ gsrc, int gT,
                    const float* __restrict__ a_scale, const float* __restrict__ b_scale, void* __restrict__ out,
                    int32_t* __restrict__ status, const FoldArgs fold) {
    static_assert(!(GATHER && FP8), "the FP8 variant reads its activation codes with TMA");
    constexpr int BN_OUT = KIND == 0 ? 128 : 256;
    constexpr int BKE = FP8 ? 128 : BK;  // K values per stage (one 128-byte swizzle row)
    constexpr int W8_BOX_BYTES = 128 * 128;  // FP8 weight box: 128 rows x 128 K codes
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    uint8_t* tiles = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    Ctl& c = *reinterpret_cast<Ctl*>(tiles + STAGES * STAGE_BYTES);
    const volatile int* abort_flag = &c.abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_tiles = (N + BN_OUT - 1) / BN_OUT;
    const int num_kb = K / BKE;
    const int kb_per = (num_kb + ksplit - 1) / ksplit;  // K blocks per slice (host: no empty slice)

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&c.full[s], GATHER ? 2 : 1);
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
        if (!GATHER) ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmA32);
        ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&c.tmem_base, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // Everything above touched only this CTA's shared and tensor memory; from here on global
    // memory written by the previous kernel is read, so wait for it (programmatic launch).
    pdl_wait();
    pdl_trigger();
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
        const int per_tile = n_tiles * ksplit;
        int sum = 0;
        if (ok)
            for (int e = e0; e < e1; ++e) sum += ((c.seg[e + 1] - c.seg[e] + BM - 1) / BM) * per_tile;
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int e = e0; e < e1; ++e) {
            c.item_start[e] = run;
            if (ok) run += ((c.seg[e + 1] - c.seg[e] + BM - 1) / BM) * per_tile;
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
            const Item it = decode_item(c, E, ksplit, swap_max, i);
            const int n0 = it.n_tile * BN_OUT;
            const int brow = it.e * K;
            const int nbox32 = (it.rows + A_BOX32_ROWS - 1) / A_BOX32_ROWS;
            // With GATHER the activation rows come from the gather warps; TMA brings the weights.
            const uint32_t tx = GATHER ? B_BYTES : (it.swap ? B_BYTES + nbox32 * A_BOX32_BYTES : STAGE_BYTES);
            const int kb0 = it.kslice * kb_per, kb1 = min(num_kb, kb0 + kb_per);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!ptx::mbar_wait(&c.empty[stage], phase ^ 1u, abort_flag)) {
                    raise_abort(c, status);
                    aborted = true;
                    break;
                }
                uint8_t* sa = tiles + stage * STAGE_BYTES;
                uint8_t* sb = sa + A_BYTES;
                // Failure-detection test hook: CTA 0 arms its first stage for 16 bytes more than its
                // copies bring, so that stage never completes and the MMA thread's bounded wait
                // must expire (status MOE_STATUS_WAIT_TIMEOUT).
                const uint32_t extra = (inject_stall && blockIdx.x == 0 && filled_mask == 0) ? 16u : 0u;
                ptx::mbar_arrive_expect_tx(&c.full[stage], tx + extra);
                if (!GATHER) {
                    if (it.swap) {
                        for (int q = 0; q < nbox32; ++q)
                            ptx::tma_load_2d(sa + q * A_BOX32_BYTES, &tmA32, &c.full[stage], kb * BKE,
                                             it.row0 + q * A_BOX32_ROWS, pol_act);
                    } else {
                        ptx::tma_load_2d(sa, &tmA, &c.full[stage], kb * BKE, it.row0, pol_act);
                    }
                }
                if (FP8) {
                    // Weight rows (output columns) of expert e: [e * 2N, e * 2N + 2N) for gate+up
                    // (gate then up), [e * N, e * N + N) for down; two 64-row blocks per box.
                    const int wrow0 = KIND == 0 ? it.e * 2 * N + n0 : it.e * N + n0;
                    const int wrow1 = KIND == 0 ? wrow0 + N : wrow0 + 128;
                    ptx::tma_load_4d(sb, &tmB, &c.full[stage], 0, 0, kb, wrow0 / 64, pol_wgt);
                    ptx::tma_load_4d(sb + W8_BOX_BYTES, &tmB, &c.full[stage], 0, 0, kb, wrow1 / 64, pol_wgt);
                } else {
#pragma unroll
                    for (int q = 0; q < B_BOXES; ++q) {
                        int col;
                        if (KIND == 0) col = (q < 2) ? n0 + q * B_BOX_N : N + n0 + (q - 2) * B_BOX_N;
                        else col = n0 + q * B_BOX_N;
                        ptx::tma_load_2d(sb + q * B_BOX_BYTES, &tmB, &c.full[stage], col, brow + kb * BK,
                                         pol_wgt);
                    }
                }
                fill_parity[stage] = phase;
                filled_mask |= 1 << stage;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (GATHER && warp >= kGatherWarp0) {
        // ------------------- gather warps (GATHER): activation rows by src[] -------------------
        // Warp g fills ring slot g each time round (positions g, g + STAGES, ... of the sequence):
        // it waits until the stage is free, issues its 128-byte rows as 16-byte cp.async copies into
        // the swizzled positions (chunk ch of tile row r at r * 128 + ((ch ^ (r & 7)) * 16)), waits
        // for its own copies, fences them for the tensor cores' (async-proxy) reads, and one lane
        // arrives on the stage's `full` barrier.  kGatherWarps stages are gathered at once.
        const int g = warp - kGatherWarp0;
        const uint64_t pol_x = ptx::policy_evict_last();  // x rows are gathered by many tiles: keep them in L2
        uint32_t stage = 0, phase = 0;
        int m = 0;  // position in the ring sequence
        bool aborted = false;
        for (int i = blockIdx.x; i < total && !aborted; i += gridDim.x) {
            const Item it = decode_item(c, E, ksplit, swap_max, i);
            const int kb0 = it.kslice * kb_per, kb1 = min(num_kb, kb0 + kb_per);
            const int nst = kb1 - kb0;
            // Does this warp fill any stage of this item?
            const int first = (g - m % kGatherWarps + kGatherWarps) % kGatherWarps;
            if (first < nst) {
                const int tile_rows = it.swap ? ((it.rows + 15) & ~15) : BM;  // rows the MMA reads
                // Lane l copies 16-byte chunk (l & 7) of tile rows (l >> 3) + 4 t: eight adjacent
                // lanes cover one 128-byte row, so each warp instruction moves four whole rows.
                const int ch = lane & 7, rs = lane >> 3;
                int tok[32];
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int r = rs + 4 * t;
                    tok[t] = r < it.rows ? __ldg(gsrc + it.row0 + r) : -1;
                    if (r < it.rows && (tok[t] < 0 || tok[t] >= gT)) {  // bad src: zero row, reported
                        flag_status(status, MOE_STATUS_BAD_SRC);
                        tok[t] = -1;
                    }
                }
                for (int j = first; j < nst; j += kGatherWarps) {
                    const int mm = m + j;
                    const uint32_t st = static_cast<uint32_t>(mm % STAGES);
                    const uint32_t ph = static_cast<uint32_t>((mm / STAGES) & 1);
                    const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(&c.empty[st], ph ^ 1u, abort_flag));
                    if (!ok) {
                        if (lane == 0) raise_abort(c, status);
                        aborted = true;
                        break;
                    }
                    const int kb = kb0 + j;
                    const uint32_t sa_u = ptx::smem_u32(tiles + st * STAGE_BYTES);
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const int r = rs + 4 * t;
                        if (r < tile_rows)
                            ptx::cp_async_16_hint(sa_u + r * 128 + ((ch ^ (r & 7)) << 4),
                                             tok[t] >= 0 ? xg + static_cast<size_t>(tok[t]) * (K / 8) + kb * 8 + ch : xg,
                                             tok[t] >= 0 ? 16u : 0u, pol_x);
                    }
                    ptx::cp_async_commit();
                    ptx::cp_async_wait_all();
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&c.full[st]);
                }
            }
            m += nst;
            (void)stage;
            (void)phase;
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------ MMA issuer ------------------------------
        constexpr uint32_t idesc_normal = ptx::idesc_bf16_f32(BM, UMMA_N, /*a_mn=*/0, /*b_mn=*/1);
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool aborted = false;
        for (int i = blockIdx.x; i < total && !aborted; i += gridDim.x) {
            const Item it = decode_item(c, E, ksplit, swap_max, i);
            const uint32_t ntok = (static_cast<uint32_t>(it.rows) + 15u) & ~15u;
            const uint32_t idesc_swap = ptx::idesc_bf16_f32(BM, ntok, /*a_mn=*/1, /*b_mn=*/0);
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
                // Activations: K-major, +32 B per 16 K.  Weights: MN-major (atoms 8 KB apart along
                // N/M, 8-row K groups 1 KB apart), +16 rows * 128 B = 2 KB per 16 K.
                const uint64_t act_desc = ptx::smem_desc_sw128(sa, 16, 1024);
                if (FP8) {
                    // Both operands K-major: +32 B (32 codes) per MMA; 8-row groups 1 KB apart.
                    const uint64_t w8_desc = ptx::smem_desc_sw128(sa + A_BYTES, 16, 1024);
                    const uint64_t w8_hi_desc = ptx::smem_desc_sw128(sa + A_BYTES + W8_BOX_BYTES, 16, 1024);
                    constexpr uint32_t idesc8_normal = ptx::idesc_e4m3_f32(BM, UMMA_N, 0, 0);
                    const uint32_t idesc8_swap = ptx::idesc_e4m3_f32(BM, ntok, 0, 0);
#pragma unroll
                    for (int kk = 0; kk < BKE / 32; ++kk) {
                        const uint32_t accum = (kb != kb0 || kk != 0) ? 1u : 0u;
                        const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
                        if (it.swap) {
                            ptx::mma_f8_ss(d_tmem, w8_desc + off, act_desc + off, idesc8_swap, accum);
                            ptx::mma_f8_ss(d_tmem + 128, w8_hi_desc + off, act_desc + off, idesc8_swap, accum);
                        } else {
                            ptx::mma_f8_ss(d_tmem, act_desc + off, w8_desc + off, idesc8_normal, accum);
                        }
                    }
                    ptx::mma_commit(&c.empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    continue;
                }
                const uint64_t wgt_desc = ptx::smem_desc_sw128(sa + A_BYTES, B_BOX_BYTES, 1024);
                const uint64_t wgt_hi_desc = ptx::smem_desc_sw128(sa + A_BYTES + 2 * B_BOX_BYTES, B_BOX_BYTES, 1024);
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                    const uint32_t accum = (kb != kb0 || kk != 0) ? 1u : 0u;
                    const uint64_t a_off = static_cast<uint64_t>((kk * 32) >> 4);
                    const uint64_t w_off = static_cast<uint64_t>((kk * 2048) >> 4);
                    if (it.swap) {
                        ptx::mma_bf16_ss(d_tmem, wgt_desc + w_off, act_desc + a_off, idesc_swap, accum);
                        ptx::mma_bf16_ss(d_tmem + 128, wgt_hi_desc + w_off, act_desc + a_off, idesc_swap, accum);
                    } else {
                        ptx::mma_bf16_ss(d_tmem, act_desc + a_off, wgt_desc + w_off, idesc_normal, accum);
                    }
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
    } else if (warp >= 2 && warp < kGatherWarp0) {
        // ------------------------------ epilogue ------------------------------
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 belong to this warp
        const int r_local = quarter * 32 + lane;
        uint32_t acc = 0, acc_phase = 0;
        for (int i = blockIdx.x; i < total; i += gridDim.x) {
            const Item it = decode_item(c, E, ksplit, swap_max, i);
            if (!ptx::mbar_wait(&c.tfull[acc], acc_phase, abort_flag)) {
                raise_abort(c, status);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * ACC_COLS;
            const int n0 = it.n_tile * BN_OUT;
            // A K-slice past the last K block (ksplit not dividing K evenly) contributes zeros.
            const bool kfull = it.kslice * kb_per < num_kb;
            if (it.swap) {
                // Accumulator lane = weight column (n0 + r_local [+128]), accumulator column = row.
                const int nchunk = (it.rows + 31) / 32;
                const int col0 = n0 + r_local;
                // FP8: column scales of this lane's two weight columns (gate/up, or col0/col0+128).
                float sc0 = 1.0f, sc1 = 1.0f;
                if (FP8) {
                    const float* sbe = b_scale + static_cast<size_t>(it.e) * (KIND == 0 ? 2 * N : N);
                    if (col0 < N) sc0 = __ldg(sbe + col0);
                    if (KIND == 0 ? col0 < N : col0 + 128 < N) sc1 = __ldg(sbe + col0 + (KIND == 0 ? N : 128));
                }
#pragma unroll 1
                for (int cc = 0; cc < nchunk; ++cc) {
                    uint32_t a0[32], a1[32];
                    ptx::tmem_ld_32x32b_x32(taddr + cc * 32, a0);
                    ptx::tmem_ld_32x32b_x32(taddr + 128 + cc * 32, a1);
                    ptx::tmem_ld_wait();
                    const int nrow = min(32, it.rows - cc * 32);
                    const size_t row_base = static_cast<size_t>(it.row0 + cc * 32);
                    if (FP8) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nrow) {
                                const float sr = __ldg(a_scale + row_base + j);  // same row in every lane
                                a0[j] = __float_as_uint(__uint_as_float(a0[j]) * (sr * sc0));
                                a1[j] = __float_as_uint(__uint_as_float(a1[j]) * (sr * sc1));
                            }
                    }
                    if (KIND == 0) {
                        uint16_t* h = reinterpret_cast<uint16_t*>(out);
                        if (col0 < N) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j < nrow)
                                    h[(row_base + j) * N + col0] =
                                        bf16_bits(silu_mul(__uint_as_float(a0[j]), __uint_as_float(a1[j])));
                        }
                    } else {
                        float* y = reinterpret_cast<float*>(out) + static_cast<size_t>(it.kslice) * M * N;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nrow) {
                                if (col0 < N) y[(row_base + j) * N + col0] = (kfull ? __uint_as_float(a0[j]) : 0.0f);
                                if (col0 + 128 < N) y[(row_base + j) * N + col0 + 128] = (kfull ? __uint_as_float(a1[j]) : 0.0f);
                            }
                    }
                }
            } else {
                // Accumulator lane = row (row0 + r_local), accumulator column = output column.
                const bool row_ok = r_local < it.rows;
                const size_t grow = static_cast<size_t>(it.row0 + r_local);
                // FP8: this lane's row scale and the expert's column scales.
                const float srow = (FP8 && row_ok) ? __ldg(a_scale + grow) : 1.0f;
                const float* sbe = FP8 ? b_scale + static_cast<size_t>(it.e) * (KIND == 0 ? 2 * N : N) : nullptr;
                if (KIND == 0) {
                    __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(out);
#pragma unroll 1
                    for (int cc = 0; cc < BN_OUT / 32; ++cc) {
                        uint32_t g[32], u[32];
                        ptx::tmem_ld_32x32b_x32(taddr + cc * 32, g);
                        ptx::tmem_ld_32x32b_x32(taddr + 128 + cc * 32, u);
                        ptx::tmem_ld_wait();
                        const int col = n0 + cc * 32;
                        if (FP8 && row_ok && col < N) {
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4) {  // the column scales are the same in every lane
                                const float4 sg = __ldg(reinterpret_cast<const float4*>(sbe + col) + j4);
                                const float4 su = __ldg(reinterpret_cast<const float4*>(sbe + N + col) + j4);
                                const float sgv[4] = {sg.x, sg.y, sg.z, sg.w}, suv[4] = {su.x, su.y, su.z, su.w};
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const int j = 4 * j4 + q;
                                    g[j] = __float_as_uint(__uint_as_float(g[j]) * (srow * sgv[q]));
                                    u[j] = __float_as_uint(__uint_as_float(u[j]) * (srow * suv[q]));
                                }
                            }
                        }
                        if (row_ok && col < N) {
                            uint4* dst = reinterpret_cast<uint4*>(h + grow * N + col);
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                uint32_t p[4];
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    p[q] = pack_bf16x2(
                                        silu_mul(__uint_as_float(g[8 * v + 2 * q]), __uint_as_float(u[8 * v + 2 * q])),
                                        silu_mul(__uint_as_float(g[8 * v + 2 * q + 1]),
                                                 __uint_as_float(u[8 * v + 2 * q + 1])));
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
                        if (FP8 && row_ok && col < N) {
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4) {
                                const float4 sc = __ldg(reinterpret_cast<const float4*>(sbe + col) + j4);
                                const float scv[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    v32[4 * j4 + q] = __float_as_uint(__uint_as_float(v32[4 * j4 + q]) * (srow * scv[q]));
                            }
                        }
                        if (row_ok && col < N) {
                            float4* dst = reinterpret_cast<float4*>(y + grow * N + col);
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                dst[v] = make_float4((kfull ? __uint_as_float(v32[4 * v]) : 0.0f),
                                                     (kfull ? __uint_as_float(v32[4 * v + 1]) : 0.0f),
                                                     (kfull ? __uint_as_float(v32[4 * v + 2]) : 0.0f),
                                                     (kfull ? __uint_as_float(v32[4 * v + 3]) : 0.0f));
                        }
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
            if (KIND == 1 && fold.cnt != nullptr) {
                // Combine fold (FoldArgs), after the accumulator is released: this thread's y stores
                // are fenced, then its rows' blocks counted.  Normal items: the thread stored 256
                // columns of its row (four 64-column blocks).  Swapped items: this warp stored the 32
                // columns n0 + 32 q.. and n0 + 128 + 32 q.. (q = its lane quarter) of every row, half
                // of two blocks; lane j % 32 counts row j once the warp's stores are fenced.
                const int n0 = it.n_tile * BN_OUT;
                const float* y0 = reinterpret_cast<const float*>(out);
                __threadfence();
                if (it.swap) {
                    __syncwarp();
                    const int bq = n0 / kFoldCols + (quarter >> 1);
                    for (int j = lane; j < it.rows; j += 32) {
                        if (n0 + 32 * quarter < N) fold_arrive(fold, y0, M, N, ksplit, it.row0 + j, bq, 1, status);
                        if (n0 + 128 + 32 * quarter < N)
                            fold_arrive(fold, y0, M, N, ksplit, it.row0 + j, bq + 128 / kFoldCols, 1, status);
                    }
                } else if (r_local < it.rows) {
                    for (int q = 0; q < BN_OUT / kFoldCols; ++q)
                        if (n0 + q * kFoldCols < N)
                            fold_arrive(fold, y0, M, N, ksplit, it.row0 + r_local, n0 / kFoldCols + q, kFoldWays, status);
                }
            }
        }
    }

    // ------------------------------ teardown ------------------------------
    if (GATHER && warp >= kGatherWarp0) ptx::cp_async_wait_all();  // no gather copy outlives the CTA
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
template <int KIND, bool GATHER, bool FP8>
cudaError_t launch_kind(const GemmArgs& a, int num_sms, cudaStream_t s, const char** why) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<KIND, GATHER, FP8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) {
            *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
            return e;
        }
        attr_set[dev] = true;
    }
    CUtensorMap mA, mA32, mB;
    const uint64_t bcols = KIND == 0 ? 2ull * a.N : static_cast<uint64_t>(a.N);
    // With GATHER, A is x [gather_T, K] (the maps over it are then unused).
    const uint64_t arows = GATHER ? static_cast<uint64_t>(a.gather_T) : static_cast<uint64_t>(a.M);
    // FP8: activation codes [M, K] and transposed weight codes [E * N_total, K], K contiguous.
    const bool maps_ok =
        FP8 ? make_tensor_map_u8(&mA, a.A, a.K, arows, BM) && make_tensor_map_u8(&mA32, a.A, a.K, arows, A_BOX32_ROWS) &&
                  make_tensor_map_w8(&mB, a.B, a.K, static_cast<uint64_t>(a.E) * bcols, 128)
            : make_tensor_map_bf16(&mA, a.A, a.K, arows, BM) &&
                  make_tensor_map_bf16(&mA32, a.A, a.K, arows, A_BOX32_ROWS) &&
                  make_tensor_map_bf16(&mB, a.B, bcols, static_cast<uint64_t>(a.E) * a.K, BK);
    if (!maps_ok) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point missing or bad operand)";
        return cudaErrorInvalidValue;
    }
    const int swap_max = a.swap_max < 0 ? 0 : (a.swap_max > SWAP_MAX_ROWS ? SWAP_MAX_ROWS : a.swap_max);
    const int ksplit = KIND == 0 ? 1 : a.ksplit;
    return launch_k(KIND == 0 ? kPdlGateUp : kPdlDown, grouped_gemm_kernel<KIND, GATHER, FP8>, dim3(num_sms),
                    dim3(GATHER ? GATHER_THREADS : NUM_THREADS), SMEM_BYTES, s, mA, mA32, mB, a.offsets, a.M, a.K,
                    a.N, a.E, ksplit, swap_max, a.inject_stall, reinterpret_cast<const int4*>(a.A), a.gather_src,
                    a.gather_T, a.a_scale, a.b_scale, a.out, a.status, a.fold);
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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
bool make_tensor_map_bf16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
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

// Blocked FP8 weight codes [rows / 64, K / 128, 64, 128] as a 4-D tensor (innermost first: 128 K
// codes, 64 rows, K block, 64-row group); box = 128 codes x 64 rows x 1 K block x box_rows / 64
// groups, which lands in shared memory as box_rows K-major rows of 128 bytes, 128-byte swizzled.
bool make_tensor_map_w8(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {128, 64, K / 128, rows / 64};
    cuuint64_t strides[3] = {128, 64 * 128, (K / 128) * 64 * 128};
    cuuint32_t box[4] = {128, 64, 1, box_rows / 64};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte tensor [rows, cols] (FP8 codes, cols contiguous), box = [box_rows, 128 cols], 128-byte swizzle.
bool make_tensor_map_u8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_grouped_gemm(int kind, const GemmArgs& a, int num_sms, cudaStream_t s,
                                const char** why) {
    if (a.ksplit < 1 || a.ksplit > kMaxKSplit || (kind == 0 && a.ksplit != 1)) {
        *why = "ksplit must be 1 for gate+up and in [1, 8] for down";
        return cudaErrorInvalidValue;
    }
    if (a.fp8 && (a.K % 128 != 0 || a.gather_src || !a.a_scale || !a.b_scale)) {
        *why = "FP8 grouped GEMM: K must be a multiple of 128, scales given, no row gather";
        return cudaErrorInvalidValue;
    }
    if (a.pair && num_sms >= 2 && !a.inject_stall) return launch_grouped_gemm_pair(kind, a, num_sms, s, why);
    if (a.fp8)
        return kind == 0 ? launch_kind<0, false, true>(a, num_sms, s, why) : launch_kind<1, false, true>(a, num_sms, s, why);
    if (kind == 0)
        return a.gather_src ? launch_kind<0, true, false>(a, num_sms, s, why)
                            : launch_kind<0, false, false>(a, num_sms, s, why);
    return launch_kind<1, false, false>(a, num_sms, s, why);
}

}  // namespace moe
