// grouped_gemm_fp8b.cu — the two grouped GEMMs of the blockwise FP8 layer on the sm_103a tensor
// cores: E4M3 operands whose scales vary along K — one per 128-wide block of an activation row and
// one per 128 x 128 block of (output column, K) of the weights, all powers of two.
//
//   kind 0: for the rows r of expert e, g[n] = sum_b P_b[r][n] * (sx[r][b] * sw[e][n/128][b]) with
//           P_b the 128-deep partial product of K block b (likewise u), h[r] = bf16(silu(g) * u);
//   kind 1: y[r][m] = sum_b P_b[r][m] * (sh[r][b] * sw[e][m/128][b]), fp32, optionally split over K.
//
// The scales do not factor out of the K sum, so the accumulation over K blocks cannot stay on the
// tensor cores: a stage is exactly one K block (128 codes, one 128-byte swizzle row), the MMA
// thread writes each block's partial product into one of two 256-column tensor-memory buffers
// (fresh, not accumulated), and eight promotion warps read it, multiply it by that block's
// scale_row * scale_col and add it into fp32 registers (a fused multiply-add: the scales are powers
// of two, so the product is exact and the add rounds once, as in the block-by-block sum it
// restates).  The item's epilogue (SwiGLU or the fp32 store) then runs from those registers.
// Blockwise FP8 is named on the HPC-Ops page; the DeepGEMM PR #304 write-up's SM100 path encodes
// its block scale factors as UE8M0 (powers of two), which these scales are.
//
// Tiles are sized for the tensor cores: one UMMA of M = 128 x N = 256 takes as long as one of
// N = 128 (measured on this kernel's hand-over loop: 0.32 us per K block either way), so every
// normal item issues N = 256 MMAs into one of two 256-column tensor-memory buffers, and eight
// promotion warps (two per tensor-memory lane quarter) each keep 128 fp32 accumulators.  For
// those registers the block's warpgroups split its register file with setmaxnreg: warpgroup 0
// (TMA producer, one or two MMA issuers, idle warps) drops to 40 registers a thread, the two
// promotion warpgroups rise to 232 (per SM sub-partition: 40 x 32 + 2 x 232 x 32 <= 16384).
//   normal   UMMA M = 128 rows x N = 256 weight columns; kind 0: gate n0..n0+127 and up
//            f+n0..f+n0+127 (128 h columns), kind 1: 256 y columns.  Weights arrive as whole
//            8 KB blocks of the blocked layout (64 rows x 128 K), 32 KB per stage.
//   swapped  (experts with at most 64 rows) UMMA M = 128 weight columns x N = rows rounded to 16,
//            two MMAs per K step (the two 128-row weight groups of the same stage) into columns
//            [0, N) and [64, 64 + N): the same weight columns as a normal item of that N-tile.
// Ring: four 48 KB stages (16 KB activations or up to 8 KB of tokens, then 32 KB of weights).
// Scheduling as in grouped_gemm.cu: (expert, N-tile, M-tile, K-slice) items, expert-major, static
// round-robin over one persistent CTA per SM.  Every wait is bounded (1 s) and reports
// MOE_STATUS_WAIT_TIMEOUT.
#include "common.cuh"
#include "fp8.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BKE = 128;                           // K codes per stage = one scale block
constexpr int STAGES = 4;
constexpr int STAGE_BYTES = 48 * 1024;
constexpr int TOK_BOX_ROWS = 32;
constexpr int TOK_BOX_BYTES = TOK_BOX_ROWS * BKE;  // 4 KB
constexpr int A_BYTES = BM * BKE;                  // 16 KB: activations, or tokens (<= 8 KB)
constexpr int WBOX128 = 128 * BKE;                 // two weight blocks, 16 KB
constexpr int W_OFF = A_BYTES;                     // weights: two 128-row groups from here
constexpr int SWAP_MAX_ROWS = 64;
constexpr int PART_COLS = 256;                     // tensor-memory columns per partial buffer
constexpr int NUM_PART = 2;
constexpr int TMEM_COLS = NUM_PART * PART_COLS;    // 512
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = 128 + 32 * EPI_WARPS;  // warp 0 TMA, warp 1 (and 2) MMA, warps 4-11 promotion
// Registers a thread: at launch (three warps per SM sub-partition: 16384 / 96 rounded down to a
// multiple of 8), then warpgroup 0 and the promotion warpgroups after setmaxnreg.  The split must
// not exceed what the block was launched with, or the increase would wait for registers forever;
// the launcher also checks the compiled count before every launch.
constexpr int REGS_LAUNCH = 168;
constexpr int REGS_CTL = 40;
constexpr int REGS_PROMO = 232;
static_assert(REGS_CTL * 128 + REGS_PROMO * 32 * EPI_WARPS <= REGS_LAUNCH * NUM_THREADS, "register split");
constexpr int MAX_E = 256;
constexpr int SMEM_BYTES = 232448;
static_assert(W_OFF + 2 * WBOX128 <= STAGE_BYTES && 2 * TOK_BOX_BYTES <= A_BYTES, "stage layout");

// Output columns of an item: kind 0 h columns, kind 1 y columns.
template <int KIND>
constexpr int bn_item() { return KIND == 0 ? 128 : 256; }

struct Ctl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t pfull[NUM_PART];   // a K block's partial product is in buffer p
    uint64_t pempty[NUM_PART];  // the promotion warps have read buffer p
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int total_items;
    int seg[MAX_E + 1];
    int item_start[MAX_E + 1];
    // Quantised h (kind 0 with h_scale): the absolute maxima of each 128-wide h block are shared
    // between the warps that hold its columns, in two slots used by alternate items.
    float xn[2][2][BM];         // normal items: [slot][half hh][row] max over the half's 64 columns
    float xs[2][2][4][32];      // swapped items: [slot][hh][lane quarter][token] max over 32 columns
    uint64_t xbar_n[2][4];      // [slot][quarter]: the quarter's two warps wrote (64 arrivals)
    uint64_t xbar_s[2][2];      // [slot][hh]: the four quarters' warps wrote (128 arrivals)
};
static_assert(STAGES * STAGE_BYTES + 1024 + sizeof(Ctl) <= SMEM_BYTES, "shared memory budget");

struct Item {
    int e, n_tile, m_tile, kslice, row0, rows;
    bool swap;
};

// Work items of an expert with cnt rows (a swapped expert takes one M-tile).
__device__ __forceinline__ int expert_items(int cnt, int N, int bn, int ksplit, int swap_max) {
    if (cnt == 0) return 0;
    const int mt = cnt <= swap_max ? 1 : (cnt + BM - 1) / BM;
    return ((N + bn - 1) / bn) * mt * ksplit;
}

// Item i: expert by binary search over item_start, then N-tile, M-tile, K-slice.
__device__ __forceinline__ Item decode_item(const Ctl& c, int E, int ksplit, int swap_max, int i) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (c.item_start[mid] <= i) lo = mid; else hi = mid;
    }
    Item it;
    it.e = lo;
    const int cnt = c.seg[lo + 1] - c.seg[lo];
    it.swap = cnt <= swap_max;
    const int mt = it.swap ? 1 : (cnt + BM - 1) / BM;
    const int j = i - c.item_start[lo];
    const int per_n = mt * ksplit;
    it.n_tile = j / per_n;
    const int r = j - it.n_tile * per_n;
    it.m_tile = r / ksplit;
    it.kslice = r - it.m_tile * ksplit;
    it.row0 = c.seg[lo] + it.m_tile * BM;
    it.rows = min(BM, cnt - it.m_tile * BM);
    return it;
}

__device__ __forceinline__ void raise_abort(Ctl& c, int32_t* status) {
    *reinterpret_cast<volatile int*>(&c.abort_flag) = 1;
    flag_status(status, MOE_STATUS_WAIT_TIMEOUT);
}

// tcgen05.wait::ld naming the 32 registers of the load it completes, so that the compiler places
// no read of them before it (a load into other registers may stay in flight across it).
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                   "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                   "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// silu(g) * u with the fast-divide intrinsic (its ~2 ulp error is far below h's bf16 rounding).
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// Two values -> two E4M3 codes (a in the low byte), rounded as to_e4m3 rounds each.
__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
    return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint16_t bf16_bits(float v) {
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&b);
}

// QH (kind 0 only): h quantised in the epilogue, a separate instance so that the plain one keeps
// its register allocation.  ALT: two MMA threads take alternate K blocks (see the MMA role).
template <int KIND, bool QH, bool ALT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_fp8b_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA32,
                         const __grid_constant__ CUtensorMap tmB128, const int32_t* __restrict__ offsets, int M,
                         int K, int N, int E, int ksplit, int swap_max, const float* __restrict__ a_scale,
                         const float* __restrict__ b_scale, void* __restrict__ out, float* __restrict__ h_scale,
                         int32_t* __restrict__ status) {
    constexpr int BN = bn_item<KIND>();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    uint8_t* tiles = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    Ctl& c = *reinterpret_cast<Ctl*>(tiles + STAGES * STAGE_BYTES);
    const volatile int* abort_flag = &c.abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int num_kb = K / BKE;
    const int kb_per = (num_kb + ksplit - 1) / ksplit;
    const int wrows = KIND == 0 ? 2 * N : N;  // weight rows (output columns) per expert
    const int nbw = wrows / 128;              // weight scale blocks per expert along N

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&c.full[s], 1);
            ptx::mbar_init(&c.empty[s], 1);
        }
        for (int p = 0; p < NUM_PART; ++p) {
            ptx::mbar_init(&c.pfull[p], 1);
            ptx::mbar_init(&c.pempty[p], EPI_WARPS);
        }
        ptx::mbar_init(&c.drain, ALT ? 2 : 1);  // one arrival per MMA thread
        for (int k = 0; k < 2; ++k) {
            for (int q = 0; q < 4; ++q) ptx::mbar_init(&c.xbar_n[k][q], 64);
            for (int q = 0; q < 2; ++q) ptx::mbar_init(&c.xbar_s[k][q], 128);
        }
        c.abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmA32);
        ptx::prefetch_tensormap(&tmB128);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&c.tmem_base, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    pdl_wait();
    pdl_trigger();
    if (warp == 2) {
        // Validate offsets and build the per-expert item prefix.
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
            for (int e = e0; e < e1; ++e) sum += expert_items(c.seg[e + 1] - c.seg[e], N, BN, ksplit, swap_max);
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int e = e0; e < e1; ++e) {
            c.item_start[e] = run;
            if (ok) run += expert_items(c.seg[e + 1] - c.seg[e], N, BN, ksplit, swap_max);
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
    uint32_t fill_parity[STAGES];
    int filled_mask = 0;

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CTL));
        if (warp == 0 && lane == 0) {
            // ------------------------------ TMA producer ------------------------------
            const uint64_t pol_act = ptx::policy_evict_last();
            const uint64_t pol_wgt = ptx::policy_evict_normal();
            uint32_t stage = 0, phase = 0;
            bool aborted = false;
            for (int i = blockIdx.x; i < total && !aborted; i += gridDim.x) {
                const Item it = decode_item(c, E, ksplit, swap_max, i);
                const int n0 = it.n_tile * BN;
                const int nbox32 = (it.rows + TOK_BOX_ROWS - 1) / TOK_BOX_ROWS;
                const uint32_t tx = (it.swap ? nbox32 * TOK_BOX_BYTES : A_BYTES) + 2 * WBOX128;
                // The two 128-row weight groups: kind 0 gate rows n0.. and up rows f+n0..; kind 1
                // output columns n0.. and n0+128.. (past the expert's last group: the next expert's
                // rows or the map's zero fill, computed and never stored).
                const int wr0 = it.e * wrows + n0;
                const int wr1 = KIND == 0 ? wr0 + N : wr0 + 128;
                const int kb0 = it.kslice * kb_per, kb1 = min(num_kb, kb0 + kb_per);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!ptx::mbar_wait(&c.empty[stage], phase ^ 1u, abort_flag)) {
                        raise_abort(c, status);
                        aborted = true;
                        break;
                    }
                    uint8_t* st = tiles + stage * STAGE_BYTES;
                    ptx::mbar_arrive_expect_tx(&c.full[stage], tx);
                    if (it.swap) {
                        for (int q = 0; q < nbox32; ++q)
                            ptx::tma_load_2d(st + q * TOK_BOX_BYTES, &tmA32, &c.full[stage], kb * BKE,
                                             it.row0 + q * TOK_BOX_ROWS, pol_act);
                    } else {
                        ptx::tma_load_2d(st, &tmA, &c.full[stage], kb * BKE, it.row0, pol_act);
                    }
                    ptx::tma_load_4d(st + W_OFF, &tmB128, &c.full[stage], 0, 0, kb, wr0 / 64, pol_wgt);
                    ptx::tma_load_4d(st + W_OFF + WBOX128, &tmB128, &c.full[stage], 0, 0, kb, wr1 / 64, pol_wgt);
                    fill_parity[stage] = phase;
                    filled_mask |= 1 << stage;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        } else if ((warp == 1 || (ALT && warp == 2)) && lane == 0) {
            // ---------------- MMA issuer: one partial product per K block, two buffers ----------------
            // ALT: the CTA's K blocks, in order over its items, alternate between the two partial
            // buffers and (four stages) between even and odd stages; warp 1 issues the even-numbered
            // blocks into buffer 0, warp 2 the odd ones into buffer 1.  A block's partial product is
            // a fresh MMA chain (nothing accumulates across blocks), so the two chains are
            // independent and every barrier still has a single MMA thread.  Each K block ends in a
            // hand-over (commit, then waits for a free partial buffer and the next stage); with two
            // threads one thread's MMAs are already queued while the other waits (gate+up, Mixtral
            // shape T=4096: 1.204 -> 1.143 ms).
            static_assert(STAGES == 2 * NUM_PART, "ALT: each thread owns one buffer and half the stages");
            const uint32_t t = ALT ? static_cast<uint32_t>(warp - 1) : 0u;
            constexpr uint32_t idesc_normal = ptx::idesc_e4m3_f32(BM, PART_COLS, 0, 0);
            uint32_t stage = t, phase = 0, pb = t, pph = 0;
            bool mine = t == 0;  // ALT: whether the next K block is this thread's
            bool aborted = false;
            for (int i = blockIdx.x; i < total && !aborted; i += gridDim.x) {
                const Item it = decode_item(c, E, ksplit, swap_max, i);
                const uint32_t ntok = (static_cast<uint32_t>(it.rows) + 15u) & ~15u;
                const uint32_t idesc_swap = ptx::idesc_e4m3_f32(BM, ntok, 0, 0);
                const int kb0 = it.kslice * kb_per, kb1 = min(num_kb, kb0 + kb_per);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (ALT) {
                        const bool m = mine;
                        mine = !mine;
                        if (!m) continue;
                    }
                    if (!ptx::mbar_wait(&c.full[stage], phase, abort_flag) ||
                        !ptx::mbar_wait(&c.pempty[pb], pph ^ 1u, abort_flag)) {
                        raise_abort(c, status);
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + pb * PART_COLS;
                    const uint32_t sa = ptx::smem_u32(tiles + stage * STAGE_BYTES);
    #pragma unroll
                    for (int kk = 0; kk < BKE / 32; ++kk) {
                        const uint32_t accum = kk != 0 ? 1u : 0u;  // a fresh partial per K block
                        const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
                        if (it.swap) {
                            // Each weight group (K-major, 128 rows) as A, the tokens (K-major) as B.
                            const uint64_t tok = ptx::smem_desc_sw128(sa, 16, 1024);
                            const uint64_t w0 = ptx::smem_desc_sw128(sa + W_OFF, 16, 1024);
                            const uint64_t w1 = ptx::smem_desc_sw128(sa + W_OFF + WBOX128, 16, 1024);
                            ptx::mma_f8_ss(d_tmem, w0 + off, tok + off, idesc_swap, accum);
                            ptx::mma_f8_ss(d_tmem + 64, w1 + off, tok + off, idesc_swap, accum);
                        } else {
                            // The activations as A, both weight groups as one 256-row B.
                            const uint64_t a = ptx::smem_desc_sw128(sa, 16, 1024);
                            const uint64_t b = ptx::smem_desc_sw128(sa + W_OFF, 16, 1024);
                            ptx::mma_f8_ss(d_tmem, a + off, b + off, idesc_normal, accum);
                        }
                    }
                    ptx::mma_commit(&c.empty[stage]);
                    ptx::mma_commit(&c.pfull[pb]);
                    if (ALT) {  // this thread's next block: two stages on, the same buffer
                        stage += 2;
                        if (stage >= STAGES) {
                            stage -= STAGES;
                            phase ^= 1u;
                        }
                        pph ^= 1u;
                    } else {
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        if (++pb == NUM_PART) {
                            pb = 0;
                            pph ^= 1u;
                        }
                    }
                }
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_PROMO));
        // ---------------- promotion + epilogue: per-block scales into fp32 registers ----------------
        // Warp w: tensor-memory lane quarter (w & 3), half hh = (w - 4) >> 2 of the buffer's columns.
        // acc[] holds 128 fp32 sums:
        //   normal kind 0: gate columns [64hh, +64) in acc[0..63], up [128 + 64hh, +64) in
        //                  acc[64..127] (the same 64 h columns);
        //   normal kind 1: columns [128hh, +128);
        //   swapped: tokens [32hh, +32) of the two MMAs, columns [32hh, +32) and [64 + 32hh, +32), in
        //            acc[0..31] and acc[32..63].
        // A K block's columns come in rounds of two 32-column loads (64 columns per wait: the
        // tensor-memory load latency, not the FMAs, sets the pace of a round).
        const int quarter = warp & 3, hh = (warp - 4) >> 2;
        const int r_local = quarter * 32 + lane;
        uint32_t pb = 0, pph = 0;
        uint32_t xn_count = 0, xs_count = 0;  // exchanges done (quantised h), per item kind
        constexpr bool quant_h = KIND == 0 && QH;
        bool aborted = false;
        for (int i = blockIdx.x; i < total && !aborted; i += gridDim.x) {
            const Item it = decode_item(c, E, ksplit, swap_max, i);
            const int n0 = it.n_tile * BN;
            const int kb0 = it.kslice * kb_per, kb1 = min(num_kb, kb0 + kb_per);
            // Weight scale blocks of the loaded columns (a block past N is computed, never stored).
            int wb0, wb1;
            if (KIND == 0) {
                wb0 = n0 / 128;
                wb1 = (N + n0) / 128;
            } else if (it.swap) {
                wb0 = n0 / 128;
                wb1 = min(nbw - 1, wb0 + 1);
            } else {
                wb0 = min(nbw - 1, (n0 + 128 * hh) / 128);
                wb1 = wb0;
            }
            const float* sw0p = b_scale + (static_cast<size_t>(it.e) * nbw + wb0) * num_kb;
            const float* sw1p = b_scale + (static_cast<size_t>(it.e) * nbw + wb1) * num_kb;
            const bool row_ok = r_local < it.rows;
            const size_t grow = static_cast<size_t>(it.row0 + r_local);
            // Does this warp hold any result column?  (Warp-uniform.)
            const bool active = it.swap ? 32 * hh < it.rows : quarter * 32 < it.rows;
            // The row / token scale this lane loads: its row (normal) or token 32hh + lane (swapped).
            const int tok = 32 * hh + lane;
            const bool sc_ok = it.swap ? tok < it.rows : row_ok;
            const float* srp =
                a_scale + (it.swap ? static_cast<size_t>(it.row0 + (sc_ok ? tok : 0)) : (sc_ok ? grow : 0)) * num_kb;
            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
            // Scales of K blocks kb (s*), kb + 1 (n*) and kb + 2 (m*): each is loaded two blocks
            // ahead of its use, so the load's latency hides behind two partial products.
            auto ld_sc = [&](int b, float& w0, float& w1, float& r) {
                const bool in = b < kb1;
                w0 = in ? __ldg(sw0p + b) : 0.0f;
                w1 = in ? __ldg(sw1p + b) : 0.0f;
                r = (in && sc_ok) ? __ldg(srp + b) : 0.0f;
            };
            float sw0, sw1, sr, nsw0, nsw1, nsr;
            ld_sc(kb0, sw0, sw1, sr);
            ld_sc(kb0 + 1, nsw0, nsw1, nsr);
            for (int kb = kb0; kb < kb1; ++kb) {
                float msw0, msw1, msr;
                ld_sc(kb + 2, msw0, msw1, msr);
                if (!ptx::mbar_wait(&c.pfull[pb], pph, abort_flag)) {
                    raise_abort(c, status);
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after();
                if (active) {
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + pb * PART_COLS;
                    uint32_t v0[32], v1[32];
                    if (it.swap) {
                        ptx::tmem_ld_32x32b_x32(taddr + 32 * hh, v0);
                        ptx::tmem_ld_32x32b_x32(taddr + 64 + 32 * hh, v1);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) {  // column j is token 32hh + j: lane j's scale
                            const float sj = __shfl_sync(0xffffffffu, sr, j);
                            acc[j] = fmaf(__uint_as_float(v0[j]), sj * sw0, acc[j]);
                            acc[32 + j] = fmaf(__uint_as_float(v1[j]), sj * sw1, acc[32 + j]);
                        }
                    } else {
                        // Four 32-column chunks, software-pipelined: chunk r + 1's load is in flight
                        // while chunk r's FMAs run (each wait names the registers it completes).
                        // kind 0: chunks gate 0..31, up 0..31, gate 32..63, up 32..63 of this warp's
                        // 64 h columns -> acc[0..], acc[64..], acc[32..], acc[96..]; kind 1:
                        // columns 32r.. of its 128 -> acc[32r..].
                        const float s0 = sr * sw0, s1 = sr * sw1;
                        auto col = [&](int r) -> uint32_t {
                            return KIND == 0 ? static_cast<uint32_t>((r & 1) * 128 + 64 * hh + 32 * (r >> 1))
                                             : static_cast<uint32_t>(128 * hh + 32 * r);
                        };
                        auto fma_chunk = [&](int r, const uint32_t (&v)[32]) {
                            const int o = KIND == 0 ? (r & 1) * 64 + (r >> 1) * 32 : 32 * r;
                            const float sc = KIND == 0 ? ((r & 1) ? s1 : s0) : s0;
#pragma unroll
                            for (int j = 0; j < 32; ++j) acc[o + j] = fmaf(__uint_as_float(v[j]), sc, acc[o + j]);
                        };
                        ptx::tmem_ld_32x32b_x32(taddr + col(0), v0);
                        tmem_ld_wait_regs(v0);
                        ptx::tmem_ld_32x32b_x32(taddr + col(1), v1);
                        fma_chunk(0, v0);
                        tmem_ld_wait_regs(v1);
                        ptx::tmem_ld_32x32b_x32(taddr + col(2), v0);
                        fma_chunk(1, v1);
                        tmem_ld_wait_regs(v0);
                        ptx::tmem_ld_32x32b_x32(taddr + col(3), v1);
                        fma_chunk(2, v0);
                        tmem_ld_wait_regs(v1);
                        fma_chunk(3, v1);
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&c.pempty[pb]);
                if (++pb == NUM_PART) {
                    pb = 0;
                    pph ^= 1u;
                }
                sw0 = nsw0;
                sw1 = nsw1;
                sr = nsr;
                nsw0 = msw0;
                nsw1 = msw1;
                nsr = msr;
            }
            if (aborted) break;
            // ------------------------------ epilogue from registers ------------------------------
            if constexpr (quant_h) {
                // h rounded to bf16 (the values the block quantiser reads), then E4M3 codes with the
                // power-of-two scale of its 128-wide block, whose absolute maximum spans two warps
                // (normal items: halves hh of the row) or four (swapped: lane quarters of a column
                // block): each warp's partial maximum goes through shared memory; a slot is rewritten
                // two items later, after every warp of the exchange has passed the next one.
                uint8_t* h8 = reinterpret_cast<uint8_t*>(out);
                const int nb = N / 128;
                if (!it.swap) {
                    float m = 0.0f;
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        acc[j] = __bfloat162float(__float2bfloat16_rn(silu_mul(acc[j], acc[64 + j])));
                        m = fmaxf(m, fabsf(acc[j]));
                    }
                    const uint32_t slot = xn_count & 1u, par = (xn_count >> 1) & 1u;
                    ++xn_count;
                    c.xn[slot][hh][r_local] = row_ok ? m : 0.0f;
                    ptx::mbar_arrive(&c.xbar_n[slot][quarter]);
                    if (!ptx::mbar_wait(&c.xbar_n[slot][quarter], par, abort_flag)) {
                        raise_abort(c, status);
                        break;
                    }
                    if (!row_ok) continue;
                    const float P = pow2_block_scale(fmaxf(m, c.xn[slot][hh ^ 1][r_local]));
                    const float inv = 1.0f / P;
                    uint4* dst = reinterpret_cast<uint4*>(h8 + grow * N + n0 + 64 * hh);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint32_t w[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int j = 16 * v + 4 * q;
                            w[q] = static_cast<uint32_t>(e4m3x2(acc[j] * inv, acc[j + 1] * inv)) |
                                   (static_cast<uint32_t>(e4m3x2(acc[j + 2] * inv, acc[j + 3] * inv)) << 16);
                        }
                        dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    if (hh == 0) h_scale[grow * nb + n0 / 128] = P;
                } else {
                    // Lane = h column n0 + r_local, acc[j] = token 32hh + j.
                    float mine = 0.0f;  // this warp's maximum for token 32hh + lane
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        acc[j] = __bfloat162float(__float2bfloat16_rn(silu_mul(acc[j], acc[32 + j])));
                        float v = fabsf(acc[j]);
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                        if (lane == j) mine = v;
                    }
                    const uint32_t slot = xs_count & 1u, par = (xs_count >> 1) & 1u;
                    ++xs_count;
                    c.xs[slot][hh][quarter][lane] = mine;
                    ptx::mbar_arrive(&c.xbar_s[slot][hh]);
                    if (!ptx::mbar_wait(&c.xbar_s[slot][hh], par, abort_flag)) {
                        raise_abort(c, status);
                        break;
                    }
                    // Lane j: the scale of token 32hh + j, then every lane takes 1/P of each token.
                    const float P = pow2_block_scale(fmaxf(fmaxf(c.xs[slot][hh][0][lane], c.xs[slot][hh][1][lane]),
                                                           fmaxf(c.xs[slot][hh][2][lane], c.xs[slot][hh][3][lane])));
                    const float inv_mine = 1.0f / P;
                    if (quarter == 0 && 32 * hh + lane < it.rows)
                        h_scale[static_cast<size_t>(it.row0 + 32 * hh + lane) * nb + n0 / 128] = P;
                    const int col = n0 + r_local;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float inv = __shfl_sync(0xffffffffu, inv_mine, j);
                        const int t = 32 * hh + j;
                        if (t < it.rows) h8[static_cast<size_t>(it.row0 + t) * N + col] = to_e4m3(acc[j] * inv);
                    }
                }
                continue;
            }
            if (!it.swap) {
                if (!row_ok) continue;
                if (KIND == 0) {
                    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + grow * N + n0 + 64 * hh);
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        uint32_t p[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            p[q] = pack_bf16x2(silu_mul(acc[8 * v + 2 * q], acc[64 + 8 * v + 2 * q]),
                                               silu_mul(acc[8 * v + 2 * q + 1], acc[64 + 8 * v + 2 * q + 1]));
                        dst[v] = make_uint4(p[0], p[1], p[2], p[3]);
                    }
                } else {
                    if (n0 + 128 * hh >= N) continue;  // the half of a last, 128-column tile past N
                    float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) +
                                                            static_cast<size_t>(it.kslice) * M * N + grow * N + n0 + 128 * hh);
#pragma unroll
                    for (int v = 0; v < 32; ++v)
                        dst[v] = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
                }
            } else {
                // Lane = weight column n0 + r_local (kind 1: and n0 + 128 + r_local), column j = token.
                const int col0 = n0 + r_local;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = 32 * hh + j;
                    if (t < it.rows) {
                        const size_t rr = static_cast<size_t>(it.row0 + t);
                        if (KIND == 0) {
                            reinterpret_cast<uint16_t*>(out)[rr * N + col0] = bf16_bits(silu_mul(acc[j], acc[32 + j]));
                        } else {
                            float* y = reinterpret_cast<float*>(out) + static_cast<size_t>(it.kslice) * M * N;
                            if (col0 < N) y[rr * N + col0] = acc[j];
                            if (col0 + 128 < N) y[rr * N + col0 + 128] = acc[32 + j];
                        }
                    }
                }
            }
        }
    }

    // ------------------------------ teardown ------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0 && c.abort_flag) {
        for (int s = 0; s < STAGES; ++s)
            if (filled_mask & (1 << s)) ptx::mbar_wait_ns(&c.full[s], fill_parity[s], 100000000ull);
    }
    if ((warp == 1 || (ALT && warp == 2)) && lane == 0) {
        ptx::mma_commit(&c.drain);
        ptx::mbar_wait_ns(&c.drain, 0, 100000000ull);
    }
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem_base, TMEM_COLS);
}

template <int KIND, bool QH, bool ALT>
cudaError_t launch_inst(const GemmArgs& a, int num_sms, cudaStream_t s, const char** why) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_fp8b_kernel<KIND, QH, ALT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) {
            *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
            return e;
        }
        attr_set[dev] = true;
    }
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, grouped_gemm_fp8b_kernel<KIND, QH, ALT>) != cudaSuccess ||
        fa.numRegs * NUM_THREADS < REGS_CTL * 128 + REGS_PROMO * 32 * EPI_WARPS) {
        *why = "blockwise FP8 GEMM: the kernel was compiled with fewer registers than its setmaxnreg split needs";
        return cudaErrorInvalidValue;
    }
    CUtensorMap mA, mA32, mB128;
    const uint64_t wrows = static_cast<uint64_t>(a.E) * (KIND == 0 ? 2ull * a.N : static_cast<uint64_t>(a.N));
    if (!make_tensor_map_u8(&mA, a.A, a.K, a.M, BM) || !make_tensor_map_u8(&mA32, a.A, a.K, a.M, TOK_BOX_ROWS) ||
        !make_tensor_map_w8(&mB128, a.B, a.K, wrows, 128)) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point missing or bad operand)";
        return cudaErrorInvalidValue;
    }
    const int swap_max = a.swap_max < 0 ? 0 : (a.swap_max > SWAP_MAX_ROWS ? SWAP_MAX_ROWS : a.swap_max);
    const int ksplit = KIND == 0 ? 1 : a.ksplit;
    return launch_k(KIND == 0 ? kPdlGateUp : kPdlDown, grouped_gemm_fp8b_kernel<KIND, QH, ALT>, dim3(num_sms),
                    dim3(NUM_THREADS), SMEM_BYTES, s, mA, mA32, mB128, a.offsets, a.M, a.K, a.N, a.E, ksplit,
                    swap_max, a.a_scale, a.b_scale, a.out, QH ? a.h_scale : nullptr, a.status);
}

// Two MMA threads (ALT) for the gate+up GEMM, and for the down GEMM when the experts average 256
// rows or more: its small-expert launches ran slower with them (Mixtral shape T=32 down 0.080 ->
// 0.089 ms, DeepSeek-V3 router 0.543 -> 0.559) while T=4096's down gained (0.627 -> 0.612).
// MOE_FP8B_ALT_ISSUE=0/1 overrides (a measurement knob).
bool fp8b_alt_issue(int kind, int M, int E) {
    if (const char* v = std::getenv("MOE_FP8B_ALT_ISSUE")) return v[0] == '1';
    return kind == 0 || static_cast<long long>(M) >= 256ll * E;
}

template <int KIND, bool QH>
cudaError_t launch_kind(const GemmArgs& a, int num_sms, cudaStream_t s, const char** why) {
    return fp8b_alt_issue(KIND, a.M, a.E) ? launch_inst<KIND, QH, true>(a, num_sms, s, why)
                                          : launch_inst<KIND, QH, false>(a, num_sms, s, why);
}

}  // namespace

cudaError_t launch_grouped_gemm_fp8b(int kind, const GemmArgs& a, int num_sms, cudaStream_t s, const char** why) {
    if (a.N % 128 != 0 || a.K % 128 != 0 || !a.a_scale || !a.b_scale) {
        *why = "blockwise FP8 grouped GEMM: N and K must be multiples of 128, scales given";
        return cudaErrorInvalidValue;
    }
    if (kind == 1) return launch_kind<1, false>(a, num_sms, s, why);
    return a.h_scale ? launch_kind<0, true>(a, num_sms, s, why) : launch_kind<0, false>(a, num_sms, s, why);
}

}  // namespace moe
