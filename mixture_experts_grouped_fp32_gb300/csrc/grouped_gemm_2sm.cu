// grouped_gemm_2sm.cu — the two grouped GEMMs of the MoE layer on pairs of SMs (tcgen05
// cta_group::2), for launches whose experts hold 128 rows or more on average.
//
// Same operations as grouped_gemm.cu, but every work item is computed by a cluster of two CTAs
// on two SMs, and one thread of CTA 0 issues M=256 UMMAs that read both CTAs' shared memory and
// accumulate into both CTAs' tensor memory.  Two item orientations:
//
//   normal  a 256-row tile of one expert: CTA r owns activation rows row0 + 128 r .. +127 (its
//           M-tile) and loads them, plus its 128-column half of the tile's 256 weight columns;
//           UMMA M = 256 rows x N = 256 weight columns (kind 0: gate and up of 128 h columns).
//           Per 64-deep K block each SM fills 32 KB of shared memory instead of the 1-SM tile's
//           48 KB, and the two M-tiles share one weight load.
//   swap    a chunk of at most C rows of one expert with the operands swapped (DeepGEMM write-up,
//           section 3.2, "dynamic swap A/B"): the weights are the UMMA A operand, M = 256 weight
//           columns (CTA r loads columns n0 + 128 r .. +127), and the tokens are B, N = rows
//           rounded up to 16 (CTA r loads its N/2 rows).  Two such UMMAs per K step, into
//           accumulator columns [0, N) and [128, 128 + N): for kind 0 gate and up, so an item
//           covers 256 h columns and one tensor-memory lane holds the gate and up value of one
//           column; for kind 1 output columns n0 + 128 r.. and n0 + 256 + 128 r.., so an item
//           covers 512 y columns.  Either way a pair streams 2 x 32 KB of weights per 64-deep K
//           block, and the MMA work is the chunk's rows, not a 256-row tile, so a small expert
//           streams its weights with the tensor pipe mostly idle.
//
// The normal-only form (SWAPCAP false) runs six 32 KB pipeline stages.  The swapping form picks
// one of two shared-memory layouts on the device, from the expert row counts, identically in
// every CTA:
//   layout A  six 32 KB stages plus a 4 KB token buffer each: chunks of C = 64 rows;
//   layout B  five 40 KB stages (32 KB + 8 KB of tokens): chunks of C = 128 rows, one stage fewer.
// Layout B is taken when some experts have 65..128 rows (swapped only under B) and they number
// at least a quarter of the normal 256-row tiles (each slowed by the shallower pipeline).  Under
// sustained load the GPU runs at its power cap, and a swapped expert's smaller MMA work raises the
// clock for everything: Mixtral shape, T=512 (3 such experts, 5 tiles) 0.544 -> 0.533 ms/layer
// with B, a skewed batch (7 experts, 2 tiles) 0.584 -> 0.523; the DeepSeek-V3 shape (5 experts,
// 61 tiles) runs best under A (2.416 vs 2.451 ms).
//   count <= min(swap_max, C)    one swapped chunk;
//   otherwise                    256-row normal tiles; a remainder of at most C rows past the last
//                                full tile becomes one swapped chunk, a larger one one more (partly
//                                empty) normal tile.
//
// Schedule.  Items are numbered expert-major; inside an expert by super tile s (the columns of a
// swapped item: normal N-tiles 2s and 2s+1), then normal items (N-tile, pair, K-slice), then the
// swapped chunk (K-slice) — items that read the same weight columns run at about the same time and
// share them through L2.  A static round-robin over the persistent grid of CTA pairs balances
// skewed loads ("Triton MoE 核心擊敗 Megablocks", setupai.cc, section 關鍵要點, block-scheduled
// grouped GEMM).  In the swapping form a swapped item reads twice the weight columns of a normal
// one, so there one schedule slot is either a swapped item or the two normal items of N-tiles 2s
// and 2s+1 for one M-tile pair, run back to back: every slot streams the same weight bytes and
// the round-robin stays balanced.  The swapping form can also split its CTA pairs between the two
// kinds of slot (see the split schedule below).
//
// Shared-memory stage (1024-byte aligned regions, 128-byte swizzle as written by TMA):
//   X (16 KB)  normal: the CTA's 128 activation rows x 64 K (K-major);
//              swap: weight boxes 0-1 (MN-major, 64 columns each, 8 KB apart)
//   Y (16 KB)  normal: the CTA's two weight boxes; swap: weight boxes 2-3 (kind 0: up)
//   T (4/8 KB) swap only: the CTA's N/2 token rows x 64 K (K-major), as 32-row boxes; after the
//              six stages in layout A, after X and Y of the stage in layout B.
//
// FP8 variant (E4M3 codes, kind::f8f6f4 pair MMAs, as in grouped_gemm.cu's FP8 instance): the
// weights are transposed, blocked codes (8 KB blocks of 64 output columns x 128 K), so each
// 64-column weight box above becomes one such block — 64 K-major rows of 128 K codes, the same
// 8 KB at the same place in shared memory — every operand is K-major,
// a stage is 128 K deep, and the epilogue multiplies by scale_row * scale_col.  Schedule, layouts
// and synchronisation are unchanged: a stage still moves the same bytes and MMA work per CTA pair
// (twice the FLOPs at twice the tensor rate).
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
constexpr int A_BYTES = BM * BK * 2;             // 16 KB: region X
constexpr int B_BOX_BYTES = 64 * BK * 2;         // 8 KB
constexpr int BH_BOXES = 2;                      // weight boxes per CTA in the normal orientation
constexpr int REGION_Y = A_BYTES;                // 16 KB
constexpr int TOK_BOX_ROWS = 32;                 // token box height in the swapped orientation
constexpr int TOK_BOX_BYTES = TOK_BOX_ROWS * BK * 2;  // 4 KB
constexpr int NORMAL_CTA_BYTES = A_BYTES + BH_BOXES * B_BOX_BYTES;  // 32 KB per CTA per stage
constexpr int STAGES_MAX = 6;
// Layout A: six 32 KB stages, then six 4 KB token buffers.  Layout B: five 40 KB stages.
constexpr int A_TOK_BASE = STAGES_MAX * NORMAL_CTA_BYTES;      // 192 KB
constexpr int B_STAGE_BYTES = NORMAL_CTA_BYTES + 2 * TOK_BOX_BYTES;  // 40 KB
constexpr int B_STAGES = 5;
constexpr int TILES_BYTES = A_TOK_BASE + STAGES_MAX * TOK_BOX_BYTES;  // 216 KB
static_assert(B_STAGES * B_STAGE_BYTES <= TILES_BYTES, "layout B fits the tile area");
constexpr int ACC_COLS = 256;
constexpr int NUM_ACC = 2;
constexpr int TMEM_COLS = NUM_ACC * ACC_COLS;
constexpr int NUM_THREADS = 192;
// GATHER launches add kGatherWarps warps (6..11) that gather the activation rows: one per
// pipeline stage, so every free stage's rows are in flight at once.
constexpr int kGatherWarps = STAGES_MAX;
constexpr int kGatherWarp0 = NUM_THREADS / 32;
constexpr int GATHER_THREADS = NUM_THREADS + 32 * kGatherWarps;
constexpr int MAX_E = 256;
constexpr int SMEM_BYTES = 232448;
// Output columns of a swapped item = of a super tile: kind 0 256 h columns (512 gate+up weight
// columns), kind 1 512 y columns; either way 2 x 32 KB of weights per pair per 64-deep K block.
template <int KIND>
constexpr int super_n() { return KIND == 0 ? 256 : 512; }
constexpr int PAIR_SWAP_MAX_ROWS = 128;
constexpr uint16_t BOTH_CTAS = 0x3;
constexpr int kMixedSplit = 1 << 20;  // split_req value selecting the proportional merge
constexpr int kAutoSplit = 1 << 21;   // split_req value: choose the split on the device
// Cost model of the automatic split (ns per pipeline stage of one CTA pair).  Gate+up: fitted to a
// sweep of the split on the DeepSeek-V3-shaped gate+up GEMM: 0.373 us per 256x256x64 pair MMA
// stage of a normal tile at the clock the tile phase runs at, 0.465 us per stage of a swapped
// chunk, which streams 2 x 32 KB of weights and is bound by the bytes one SM pair keeps in flight.
// Down: a normal stage costs about as much as a swapped one (0.470 us): its items are only
// d_ff / 64 stages deep, so the accumulator hand-over and the 128 KB fp32 epilogue of every item
// weigh more; fitted to the per-pair finishing times of both DeepSeek-shaped down GEMMs (CTA
// pairs of each kind busy until the same time at P = 57 with DeepSeek-V3's router and P = 45 with
// the softmax router, against 53 and 41 with the gate+up costs).
template <int KIND>
constexpr long long normal_stage_ns() { return KIND == 0 ? 373 : 470; }
constexpr long long kSwapStageNs = 465;

template <bool SWAPCAP>
struct Cfg {
    static constexpr int TILES = SWAPCAP ? TILES_BYTES : STAGES_MAX * NORMAL_CTA_BYTES;
};

struct Ctl {
    uint64_t full[STAGES_MAX];
    uint64_t empty[STAGES_MAX];
    uint64_t tfull[NUM_ACC];
    uint64_t tempty[NUM_ACC];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int total_items;
    int layout_b;  // swapping form: 1 = layout B (five 40 KB stages, 128-row chunks)
    int split_p;   // split schedule: pairs [0, split_p) run normal slots, the rest swapped ones; 0 = off
    int total_normal;
    int seg[MAX_E + 1];
    int item_start[MAX_E + 1];  // round-robin: first slot of each expert; split: first swapped slot
    int nstart[MAX_E + 1];      // split: first normal slot of each expert
};
static_assert(Cfg<true>::TILES + 1024 + sizeof(Ctl) <= SMEM_BYTES, "shared memory budget");

// Pipeline geometry of one launch (uniform across the grid).
struct Ring {
    int nst, stride, chunk;  // stages, stage stride in bytes, swapped-chunk rows (C)
    __device__ __forceinline__ uint32_t tok_off(int s) const {
        return chunk > 64 ? static_cast<uint32_t>(s * stride + NORMAL_CTA_BYTES)
                          : static_cast<uint32_t>(A_TOK_BASE + s * TOK_BOX_BYTES);
    }
};
template <bool SWAPCAP>
__device__ __forceinline__ Ring make_ring(int layout_b) {
    if (SWAPCAP && layout_b) return Ring{B_STAGES, B_STAGE_BYTES, 128};
    return Ring{STAGES_MAX, NORMAL_CTA_BYTES, 64};
}

// How an expert's rows split into normal 256-row pair tiles (np) and at most one swapped chunk
// (ns, starting at row sbase of the expert).
struct RowSplit {
    int np, ns, sbase;
};
template <bool SWAPCAP>
__device__ __forceinline__ RowSplit split_rows(int cnt, int swap_max, int chunk) {
    RowSplit s{0, 0, 0};
    if (cnt <= 0) return s;
    if (!SWAPCAP) {
        s.np = (cnt + 2 * BM - 1) / (2 * BM);
    } else if (cnt <= min(swap_max, chunk)) {
        s.ns = 1;
    } else {
        s.np = cnt / (2 * BM);
        const int rem = cnt - 2 * BM * s.np;
        if (rem > chunk || (rem > 0 && s.np == 0)) {
            ++s.np;
        } else if (rem > 0) {
            s.ns = 1;
            s.sbase = 2 * BM * s.np;
        }
    }
    return s;
}

// Column tiling of one launch.  Normal N-tiles are BN_OUT output columns (kind 0: 128 h columns,
// kind 1: 256 y columns); R = 2 of them make one super tile (the columns of a swapped item); the
// last super tile may hold fewer (r_last).
template <int KIND>
struct Tiling {
    int n_super, r_last;
    static constexpr int BN_OUT = KIND == 0 ? 128 : 256;
    static constexpr int R = super_n<KIND>() / BN_OUT;
    __device__ __forceinline__ explicit Tiling(int N) {
        const int n_tiles = (N + BN_OUT - 1) / BN_OUT;
        n_super = (n_tiles + R - 1) / R;
        r_last = n_tiles - R * (n_super - 1);
    }
};

// Whether one schedule slot holds the normal items of a whole super tile (see the header).
template <int KIND, bool SWAPCAP>
struct Sched {
    static constexpr bool GROUP = SWAPCAP;
};

template <int KIND, bool SWAPCAP>
__device__ __forceinline__ int expert_items(int cnt, const Tiling<KIND>& t, int ksplit, int swap_max, int chunk) {
    const RowSplit s = split_rows<SWAPCAP>(cnt, swap_max, chunk);
    if (Sched<KIND, SWAPCAP>::GROUP) return t.n_super * (s.np + s.ns) * ksplit;
    return ((t.n_super - 1) * (Tiling<KIND>::R * s.np + s.ns) + (t.r_last * s.np + s.ns)) * ksplit;
}

struct PairItem {
    int e, n_tile, kslice, row0, rows;  // normal: this CTA's M-tile (rows may be <= 0)
    int swap, ntok;                     // swap: row0/rows = the chunk, ntok = rows rounded to 16
    int nsub;                           // items in this slot: N-tiles n_tile .. n_tile + nsub - 1
};

template <int KIND, bool SWAPCAP>
__device__ __forceinline__ PairItem decode_pair_item(const Ctl& c, const Tiling<KIND>& t, int E, int ksplit,
                                                     int swap_max, int chunk, int rank, int i) {
    int lo = 0, hi = E;  // item_start[lo] <= i < item_start[lo + 1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (c.item_start[mid] <= i) lo = mid; else hi = mid;
    }
    PairItem it;
    it.e = lo;
    const int cnt = c.seg[lo + 1] - c.seg[lo];
    const RowSplit s = split_rows<SWAPCAP>(cnt, swap_max, chunk);
    constexpr int R = Tiling<KIND>::R;
    constexpr bool GROUP = Sched<KIND, SWAPCAP>::GROUP;
    const int per_full = ((GROUP ? 1 : R) * s.np + s.ns) * ksplit;
    const int j = i - c.item_start[lo];
    const int st = min(j / per_full, t.n_super - 1);
    const int r = j - st * per_full;
    const int rs = st == t.n_super - 1 ? t.r_last : R;
    const int n_normal = (GROUP ? 1 : rs) * s.np * ksplit;
    it.nsub = 1;
    if (r < n_normal) {
        const int per_n = s.np * ksplit;
        const int ntl = r / per_n;  // 0 when GROUP
        const int rr = r - ntl * per_n;
        const int mpair = rr / ksplit;
        it.kslice = rr - mpair * ksplit;
        it.n_tile = R * st + ntl;
        if (GROUP) it.nsub = rs;
        const int mtile = 2 * mpair + rank;
        it.row0 = c.seg[lo] + mtile * BM;
        it.rows = min(BM, cnt - mtile * BM);
        it.swap = 0;
        it.ntok = 0;
    } else {
        it.kslice = r - n_normal;  // the only chunk
        it.n_tile = st;
        it.row0 = c.seg[lo] + s.sbase;
        it.rows = min(chunk, cnt - s.sbase);
        it.swap = 1;
        it.ntok = (it.rows + 15) & ~15;
    }
    return it;
}

// Split schedule (swapping form only).  In a many-expert layer the large experts' normal tiles are
// bound by the tensor pipe (2+ tile pairs reuse their weights from L2) and the small experts'
// swapped chunks by the weight bytes a pair keeps in flight; one round-robin in expert order runs
// the two kinds one after the other.  Instead, P CTA pairs run the normal slots and the others the
// swapped slots, at the same time; P comes from a cost model of both kinds' work, evaluated on the
// device from the row counts (kernel argument split_req: 0 off, P, kMixedSplit, kAutoSplit).  For
// this the normal slots and the swapped slots are numbered separately, each expert-major.  Normal slot numbering inside an expert: super tile, M-tile pair,
// K-slice (kind 0: one slot = N-tiles 2s and 2s+1, as in the round-robin order); swapped: super
// tile, K-slice.
template <int KIND>
__device__ __forceinline__ int expert_normal_slots(int cnt, const Tiling<KIND>& t, int ksplit, int swap_max,
                                                   int chunk) {
    const RowSplit s = split_rows<true>(cnt, swap_max, chunk);
    return t.n_super * s.np * ksplit;
}
template <int KIND>
__device__ __forceinline__ int expert_swap_slots(int cnt, const Tiling<KIND>& t, int ksplit, int swap_max,
                                                 int chunk) {
    return t.n_super * split_rows<true>(cnt, swap_max, chunk).ns * ksplit;
}

template <int KIND>
__device__ __forceinline__ PairItem decode_split_item(const Ctl& c, const Tiling<KIND>& t, int E, int ksplit,
                                                      int swap_max, int chunk, int rank, bool normal, int i) {
    const int* start = normal ? c.nstart : c.item_start;
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (start[mid] <= i) lo = mid; else hi = mid;
    }
    PairItem it;
    it.e = lo;
    const int cnt = c.seg[lo + 1] - c.seg[lo];
    const RowSplit s = split_rows<true>(cnt, swap_max, chunk);
    const int j = i - start[lo];
    it.nsub = 1;
    if (normal) {
        const int per_st = s.np * ksplit;
        const int st = j / per_st;
        const int r = j - st * per_st;
        const int mpair = r / ksplit;
        it.kslice = r - mpair * ksplit;
        it.n_tile = Tiling<KIND>::R * st;
        it.nsub = st == t.n_super - 1 ? t.r_last : Tiling<KIND>::R;
        const int mtile = 2 * mpair + rank;
        it.row0 = c.seg[lo] + mtile * BM;
        it.rows = min(BM, cnt - mtile * BM);
        it.swap = 0;
        it.ntok = 0;
    } else {
        const int st = j / ksplit;
        it.kslice = j - st * ksplit;
        it.n_tile = st;
        it.row0 = c.seg[lo] + s.sbase;
        it.rows = min(chunk, cnt - s.sbase);
        it.swap = 1;
        it.ntok = (it.rows + 15) & ~15;
    }
    return it;
}

// The slots one CTA pair runs: `count` slots first, first + stride, ... of one numbering.
struct Walk {
    int first, stride, count, mode;  // mode 0 round-robin over all slots, 1 normal, 2 swapped,
                                     // 3 round-robin over the proportional merge of both
};

// Mixed order (mode 3): the normal and the swapped slots merged in proportion to their counts
// (n_normal : n_swap), slot i of the merge being normal iff floor((i+1) n / t) > floor(i n / t) —
// so every CTA pair of the round-robin gets the same share of each kind, and spends time on each
// in proportion to its work: tensor-bound tiles and weight streams run side by side on the GPU.
__device__ __forceinline__ void mixed_slot(int i, int n_normal, int n_total, bool* normal, int* idx) {
    const long long a = static_cast<long long>(i) * n_normal / n_total;
    const long long b = static_cast<long long>(i + 1) * n_normal / n_total;
    *normal = b > a;
    *idx = *normal ? static_cast<int>(a) : i - static_cast<int>(a);
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

// GATHER (kind 0 only): each CTA's six extra warps gather its own activation rows from x by
// src[] with cp.async, as in grouped_gemm.cu; CTA 0's `full` barrier then expects three arrivals:
// the TMA weight bytes', and one per CTA when its gathered rows have landed (CTA 1's remotely).
template <int KIND, bool SWAPCAP, bool GATHER, bool FP8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GATHER ? GATHER_THREADS : NUM_THREADS, 1)
grouped_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA32,
                        const __grid_constant__ CUtensorMap tmB, const int32_t* __restrict__ offsets, int M,
                        int K, int N, int E, int ksplit, int swap_max, int layout_mode, int split_req,
                        const int4* __restrict__ xg, const int32_t* __restrict__ gsrc, int gT,
                        const float* __restrict__ a_scale, const float* __restrict__ b_scale, void* __restrict__ out,
                        int32_t* __restrict__ status, const FoldArgs fold) {
    static_assert(!(GATHER && FP8), "the FP8 variant reads its activation codes with TMA");
    constexpr int BN_OUT = Tiling<KIND>::BN_OUT;
    constexpr int BKE = FP8 ? 128 : BK;  // K values per stage (one 128-byte swizzle row)
    const int wrows = KIND == 0 ? 2 * N : N;  // FP8: weight rows (output columns) per expert
    constexpr int SW_BOXES = 4;  // weight boxes per CTA in a swapped item (two MMAs)
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    uint8_t* tiles = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    Ctl& c = *reinterpret_cast<Ctl*>(tiles + Cfg<SWAPCAP>::TILES);
    const volatile int* abort_flag = &c.abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = static_cast<int>(ptx::cluster_ctarank());
    const bool leader = rank == 0;
    const int pair_id = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
    const Tiling<KIND> tiling(N);
    const int num_kb = K / BKE;
    const int kb_per = (num_kb + ksplit - 1) / ksplit;

    if (tid == 0) {
        for (int s = 0; s < STAGES_MAX; ++s) {
            ptx::mbar_init(&c.full[s], GATHER ? 3 : 1);
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
        if (!GATHER) ptx::prefetch_tensormap(&tmA);
        if (SWAPCAP && !GATHER) ptx::prefetch_tensormap(&tmA32);
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
        // Layout choice (swapping form): B when there are experts that only B swaps (65..128
        // rows) and they number at least a quarter of the normal 256-row tiles B slows down.
        int layout_b = 0;
        if (SWAPCAP && ok) {
            int mid = 0, tiles_b = 0;
            for (int e = e0; e < e1; ++e) {
                const int cnt = c.seg[e + 1] - c.seg[e];
                mid += (cnt > 64 && cnt <= min(swap_max, 128)) ? 1 : 0;
                tiles_b += split_rows<SWAPCAP>(cnt, swap_max, 128).np;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                mid += __shfl_xor_sync(0xffffffffu, mid, o);
                tiles_b += __shfl_xor_sync(0xffffffffu, tiles_b, o);
            }
            layout_b = (mid > 0 && 4 * mid >= tiles_b) ? 1 : 0;
        }
        if (SWAPCAP && layout_mode != 0) layout_b = layout_mode == 2 ? 1 : 0;  // host override
        const int chunk = make_ring<SWAPCAP>(layout_b).chunk;
        // Split schedule: only when both kinds of slot exist.
        int nsum = 0, ssum = 0;
        if (SWAPCAP && split_req != 0 && ok)
            for (int e = e0; e < e1; ++e) {
                const int cnt = c.seg[e + 1] - c.seg[e];
                nsum += expert_normal_slots<KIND>(cnt, tiling, ksplit, swap_max, chunk);
                ssum += expert_swap_slots<KIND>(cnt, tiling, ksplit, swap_max, chunk);
            }
        int ntot = nsum, stot = ssum;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            ntot += __shfl_xor_sync(0xffffffffu, ntot, o);
            stot += __shfl_xor_sync(0xffffffffu, stot, o);
        }
        // Automatic split: P pairs for the normal tiles, in proportion to the modelled work of each
        // kind.  Only when each kind is at least 15 % of it (otherwise one round-robin overlaps the
        // little there is of the other kind well enough), and when most normal-tile stages belong
        // to experts with two or more pair tiles — those reuse their weights from L2 and are bound
        // by the tensor pipe; a one-tile expert streams its weights like a swapped chunk, and with
        // both kinds memory-bound a split only unbalances the bytes (Mixtral T=512: +5 %).
        int auto_p = 0;
        if (SWAPCAP && split_req == kAutoSplit && ok) {
            long long hs = 0, hs_reuse = 0, ls = 0;  // pair-stages: normal tiles, of them reused, swapped
            const int n_tiles = (N + Tiling<KIND>::BN_OUT - 1) / Tiling<KIND>::BN_OUT;
            for (int e = e0; e < e1; ++e) {
                const RowSplit rs = split_rows<true>(c.seg[e + 1] - c.seg[e], swap_max, chunk);
                const long long h = static_cast<long long>(rs.np) * n_tiles * num_kb;
                hs += h;
                hs_reuse += rs.np >= 2 ? h : 0;
                ls += static_cast<long long>(rs.ns) * tiling.n_super * num_kb;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                hs += __shfl_xor_sync(0xffffffffu, hs, o);
                hs_reuse += __shfl_xor_sync(0xffffffffu, hs_reuse, o);
                ls += __shfl_xor_sync(0xffffffffu, ls, o);
            }
            const long long wh = hs * normal_stage_ns<KIND>(), wl = ls * kSwapStageNs, wt = wh + wl;
            if (wt > 0 && 100 * wh >= 15 * wt && 100 * wl >= 15 * wt && 2 * hs_reuse >= hs) {
                auto_p = static_cast<int>((2 * num_pairs * wh + wt) / (2 * wt));  // rounded
                auto_p = max(1, min(num_pairs - 1, auto_p));
            }
        }
        const int req = split_req == kAutoSplit ? auto_p : split_req;
        const bool split = SWAPCAP && req > 0 && ok && ntot > 0 && stot > 0 &&
                           (num_pairs >= 2 || req == kMixedSplit);
        // Exclusive scans: round-robin slots into item_start; or normal slots into nstart and
        // swapped slots into item_start.
        int sum = 0;
        if (ok && !split)
            for (int e = e0; e < e1; ++e)
                sum += expert_items<KIND, SWAPCAP>(c.seg[e + 1] - c.seg[e], tiling, ksplit, swap_max, chunk);
        if (split) sum = ssum;
        int incl = sum, nincl = nsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            const int nv = __shfl_up_sync(0xffffffffu, nincl, o);
            if (lane >= o) {
                incl += v;
                nincl += nv;
            }
        }
        int run = incl - sum, nrun = nincl - nsum;
        for (int e = e0; e < e1; ++e) {
            const int cnt = c.seg[e + 1] - c.seg[e];
            c.item_start[e] = run;
            c.nstart[e] = nrun;
            if (split) {
                run += expert_swap_slots<KIND>(cnt, tiling, ksplit, swap_max, chunk);
                nrun += expert_normal_slots<KIND>(cnt, tiling, ksplit, swap_max, chunk);
            } else if (ok) {
                run += expert_items<KIND, SWAPCAP>(cnt, tiling, ksplit, swap_max, chunk);
            }
        }
        if (lane == 31) {
            c.item_start[E] = incl;
            c.nstart[E] = nincl;
            c.total_items = incl;
            c.total_normal = split ? nincl : 0;
            c.split_p = split ? (req == kMixedSplit ? kMixedSplit : min(req, num_pairs - 1)) : 0;
            c.layout_b = layout_b;
        }
        if (!ok && lane == 0 && leader) flag_status(status, MOE_STATUS_BAD_OFFSETS);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrive or copy
    ptx::tc_fence_after();

    const uint32_t tmem_base = c.tmem_base;
    const Ring ring = make_ring<SWAPCAP>(c.layout_b);
    const int chunk = ring.chunk;
    Walk walk{pair_id, num_pairs, c.total_items, 0};
    if (c.split_p == kMixedSplit)
        walk = Walk{pair_id, num_pairs, c.total_normal + c.total_items, 3};
    else if (c.split_p > 0)
        walk = pair_id < c.split_p ? Walk{pair_id, c.split_p, c.total_normal, 1}
                                   : Walk{pair_id - c.split_p, num_pairs - c.split_p, c.total_items, 2};
    auto slot_at = [&](int i) {
        if (walk.mode == 0) return decode_pair_item<KIND, SWAPCAP>(c, tiling, E, ksplit, swap_max, chunk, rank, i);
        bool normal = walk.mode == 1;
        int j = i;
        if (walk.mode == 3) mixed_slot(i, c.total_normal, walk.count, &normal, &j);
        return decode_split_item<KIND>(c, tiling, E, ksplit, swap_max, chunk, rank, normal, j);
    };
    uint32_t fill_parity[STAGES_MAX];
    int filled_mask = 0;

    if (warp == 0 && lane == 0) {
        // ------------------------------ TMA producer (both CTAs) ------------------------------
        const uint64_t pol_act = ptx::policy_evict_last();
        const uint64_t pol_wgt = ptx::policy_evict_normal();
        int stage = 0;
        uint32_t phase = 0;
        bool aborted = false;
        for (int i = walk.first; i < walk.count && !aborted; i += walk.stride) {
          const PairItem slot = slot_at(i);
          for (int sub = 0; sub < slot.nsub && !aborted; ++sub) {
            PairItem it = slot;
            it.n_tile += sub;
            const int brow = it.e * K;
            const int kb0 = it.kslice * kb_per, kb1 = min(num_kb, kb0 + kb_per);
            // Swapped items: this CTA's token rows start N/2 into the chunk for CTA 1.
            const int half = it.ntok >> 1;
            const int ntb = (half + TOK_BOX_ROWS - 1) / TOK_BOX_ROWS;  // 1 (layout A) or up to 2 (B)
            // With GATHER the activation rows come from the gather warps; TMA brings the weights.
            const uint32_t pair_tx = GATHER ? (it.swap ? 2u * SW_BOXES * B_BOX_BYTES : 2u * BH_BOXES * B_BOX_BYTES)
                                            : (it.swap ? 2u * (SW_BOXES * B_BOX_BYTES + ntb * TOK_BOX_BYTES)
                                                       : 2u * NORMAL_CTA_BYTES);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!ptx::mbar_wait(&c.empty[stage], phase ^ 1u, abort_flag)) {
                    raise_abort(c, status);
                    aborted = true;
                    break;
                }
                uint8_t* sa = tiles + stage * ring.stride;
                const uint32_t full_leader = ptx::map_to_cta(ptx::smem_u32(&c.full[stage]), 0);
                if (leader) ptx::mbar_arrive_expect_tx(&c.full[stage], pair_tx);
                if (SWAPCAP && it.swap) {
                    const int n0 = it.n_tile * super_n<KIND>() + 128 * rank;
                    if (!GATHER) {
                        uint8_t* st = tiles + ring.tok_off(stage);
                        for (int q = 0; q < ntb; ++q)
                            ptx::tma_load_2d_pair(st + q * TOK_BOX_BYTES, &tmA32, full_leader, kb * BKE,
                                                  it.row0 + rank * half + q * TOK_BOX_ROWS, pol_act);
                    }
#pragma unroll
                    for (int q = 0; q < SW_BOXES; ++q) {
                        // kind 0: gate n0, n0+64, up f+n0, f+n0+64; kind 1: n0, n0+64, n0+256, n0+320.
                        // (FP8: the same output columns as 64-row boxes of the transposed codes.)
                        const int col = q < 2 ? n0 + 64 * q : (KIND == 0 ? N : 256) + n0 + 64 * (q - 2);
                        if (FP8)
                            ptx::tma_load_4d_pair(sa + q * B_BOX_BYTES, &tmB, full_leader, 0, 0, kb,
                                                  (it.e * wrows + col) / 64, pol_wgt);
                        else
                            ptx::tma_load_2d_pair(sa + q * B_BOX_BYTES, &tmB, full_leader, col, brow + kb * BK,
                                                  pol_wgt);
                    }
                } else {
                    const int n0 = it.n_tile * BN_OUT;
                    if (!GATHER) ptx::tma_load_2d_pair(sa, &tmA, full_leader, kb * BKE, it.row0, pol_act);
#pragma unroll
                    for (int q = 0; q < BH_BOXES; ++q) {
                        // kind 0: CTA r holds gate columns n0+64r.. and up columns f+n0+64r..;
                        // kind 1: CTA r holds output columns n0+128r .. n0+128r+127.
                        const int col = KIND == 0 ? (q == 0 ? n0 + 64 * rank : N + n0 + 64 * rank)
                                                  : n0 + 128 * rank + 64 * q;
                        if (FP8)
                            ptx::tma_load_4d_pair(sa + REGION_Y + q * B_BOX_BYTES, &tmB, full_leader, 0, 0, kb,
                                                  (it.e * wrows + col) / 64, pol_wgt);
                        else
                            ptx::tma_load_2d_pair(sa + REGION_Y + q * B_BOX_BYTES, &tmB, full_leader, col,
                                                  brow + kb * BK, pol_wgt);
                    }
                }
                fill_parity[stage] = phase;
                filled_mask |= 1 << stage;
                if (++stage == ring.nst) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
          }
        }
    } else if (GATHER && warp >= kGatherWarp0) {
        // ------------------- gather warps (GATHER, both CTAs): activation rows by src[] -------------------
        // As in grouped_gemm.cu: warp g fills ring slot g each time round (positions g, g + stages,
        // ... of the ring sequence) with this CTA's rows (normal: its 128-row M-tile; swapped: its
        // N/2 token rows), waits for its own copies, fences them, and one lane arrives on CTA 0's
        // `full` barrier of the stage (CTA 1 remotely).
        const int g = warp - kGatherWarp0;
        const uint64_t pol_x = ptx::policy_evict_last();  // x rows are gathered by many tiles: keep them in L2
        int m = 0;  // position in the ring sequence
        bool aborted = false;
        for (int i = walk.first; i < walk.count && !aborted; i += walk.stride) {
          const PairItem slot = slot_at(i);
          for (int sub = 0; sub < slot.nsub && !aborted; ++sub) {
            PairItem it = slot;
            it.n_tile += sub;
            const int kb0 = it.kslice * kb_per, kb1 = min(num_kb, kb0 + kb_per);
            const int nst = kb1 - kb0;
            // Warp g owns ring slot g: positions mm with mm % stages == g.  One warp per slot keeps
            // every waiter on a slot's `empty` barrier at most one phase ahead, which its parity wait
            // needs (warps g >= stages have nothing to do).
            const int first = (g - m % ring.nst + ring.nst) % ring.nst;
            if (g < ring.nst && first < nst) {
                const int half = it.ntok >> 1;
                const int tile_rows = it.swap ? half : BM;
                // Lane l copies 16-byte chunk (l & 7) of tile rows (l >> 3) + 4 t: eight adjacent
                // lanes cover one 128-byte row, so each warp instruction moves four whole rows.
                const int ch = lane & 7, rs = lane >> 3;
                int tok[32];
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int r = rs + 4 * t;
                    const int rr = it.swap ? rank * half + r : r;  // row within the item's rows
                    const bool valid = r < tile_rows && rr < it.rows;
                    tok[t] = valid ? __ldg(gsrc + it.row0 + (it.swap ? rank * half : 0) + r) : -1;
                    if (valid && (tok[t] < 0 || tok[t] >= gT)) {  // bad src: zero row, reported
                        flag_status(status, MOE_STATUS_BAD_SRC);
                        tok[t] = -1;
                    }
                }
                for (int j = first; j < nst; j += ring.nst) {
                    const int mm = m + j;
                    const int st = mm % ring.nst;  // == g
                    const uint32_t ph = static_cast<uint32_t>((mm / ring.nst) & 1);
                    const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(&c.empty[st], ph ^ 1u, abort_flag));
                    if (!ok) {
                        if (lane == 0) raise_abort(c, status);
                        aborted = true;
                        break;
                    }
                    const int kb = kb0 + j;
                    const uint32_t dst = ptx::smem_u32(it.swap ? tiles + ring.tok_off(st) : tiles + st * ring.stride);
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const int r = rs + 4 * t;
                        if (r < tile_rows)
                            ptx::cp_async_16_hint(dst + r * 128 + ((ch ^ (r & 7)) << 4),
                                             tok[t] >= 0 ? xg + static_cast<size_t>(tok[t]) * (K / 8) + kb * 8 + ch : xg,
                                             tok[t] >= 0 ? 16u : 0u, pol_x);
                    }
                    ptx::cp_async_commit();
                    ptx::cp_async_wait_all();
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (leader) ptx::mbar_arrive(&c.full[st]);
                        else ptx::mbar_arrive_cluster(ptx::map_to_cta(ptx::smem_u32(&c.full[st]), 0));
                    }
                }
            }
            m += nst;
          }
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------ pair MMA issuer (CTA 0) ------------------------------
        constexpr uint32_t idesc_normal = FP8 ? ptx::idesc_e4m3_f32(2 * BM, ACC_COLS, 0, 0)
                                              : ptx::idesc_bf16_f32(2 * BM, ACC_COLS, /*a_mn=*/0, /*b_mn=*/1);
        int stage = 0;
        uint32_t phase = 0, acc = 0, acc_phase = 0;
        bool aborted = false;
        for (int i = walk.first; i < walk.count && !aborted; i += walk.stride) {
          const PairItem slot = slot_at(i);
          for (int sub = 0; sub < slot.nsub && !aborted; ++sub) {
            const PairItem& it = slot;
            const uint32_t idesc_swap = FP8 ? ptx::idesc_e4m3_f32(2 * BM, static_cast<uint32_t>(it.ntok), 0, 0)
                                            : ptx::idesc_bf16_f32(2 * BM, static_cast<uint32_t>(it.ntok), 1, 0);
            const int kb0 = it.kslice * kb_per, kb1 = min(num_kb, kb0 + kb_per);
            if (!ptx::mbar_wait(&c.tempty[acc], acc_phase ^ 1u, abort_flag)) {
                raise_abort(c, status);
                aborted = true;
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
                const uint32_t sa = ptx::smem_u32(tiles + stage * ring.stride);
                if (FP8) {
                    // Every operand K-major: +32 B (32 codes) per MMA, 8-row groups 1 KB apart.
                    if (SWAPCAP && it.swap) {
                        const uint64_t wx_desc = ptx::smem_desc_sw128(sa, 16, 1024);
                        const uint64_t wy_desc = ptx::smem_desc_sw128(sa + REGION_Y, 16, 1024);
                        const uint64_t tok_desc = ptx::smem_desc_sw128(ptx::smem_u32(tiles + ring.tok_off(stage)), 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < BKE / 32; ++kk) {
                            const uint32_t accum = (kb != kb0 || kk != 0) ? 1u : 0u;
                            const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
                            ptx::mma_f8_ss_pair(d_tmem, wx_desc + off, tok_desc + off, idesc_swap, accum);
                            ptx::mma_f8_ss_pair(d_tmem + 128, wy_desc + off, tok_desc + off, idesc_swap, accum);
                        }
                    } else {
                        const uint64_t a_desc = ptx::smem_desc_sw128(sa, 16, 1024);
                        const uint64_t b_desc = ptx::smem_desc_sw128(sa + REGION_Y, 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < BKE / 32; ++kk) {
                            const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
                            ptx::mma_f8_ss_pair(d_tmem, a_desc + off, b_desc + off, idesc_normal,
                                                (kb != kb0 || kk != 0) ? 1u : 0u);
                        }
                    }
                } else if (SWAPCAP && it.swap) {
                    // Weights MN-major (A, 64-column atoms 8 KB apart), tokens K-major (B).
                    const uint64_t wx_desc = ptx::smem_desc_sw128(sa, B_BOX_BYTES, 1024);
                    const uint64_t wy_desc = ptx::smem_desc_sw128(sa + REGION_Y, B_BOX_BYTES, 1024);
                    const uint64_t tok_desc = ptx::smem_desc_sw128(ptx::smem_u32(tiles + ring.tok_off(stage)), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        const uint32_t accum = (kb != kb0 || kk != 0) ? 1u : 0u;
                        const uint64_t w_off = static_cast<uint64_t>((kk * 2048) >> 4);
                        const uint64_t t_off = static_cast<uint64_t>((kk * 32) >> 4);
                        ptx::mma_bf16_ss_pair(d_tmem, wx_desc + w_off, tok_desc + t_off, idesc_swap, accum);
                        ptx::mma_bf16_ss_pair(d_tmem + 128, wy_desc + w_off, tok_desc + t_off, idesc_swap, accum);
                    }
                } else {
                    const uint64_t a_desc = ptx::smem_desc_sw128(sa, 16, 1024);
                    const uint64_t b_desc = ptx::smem_desc_sw128(sa + REGION_Y, B_BOX_BYTES, 1024);
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)
                        ptx::mma_bf16_ss_pair(d_tmem, a_desc + static_cast<uint64_t>((kk * 32) >> 4),
                                              b_desc + static_cast<uint64_t>((kk * 2048) >> 4), idesc_normal,
                                              (kb != kb0 || kk != 0) ? 1u : 0u);
                }
                ptx::mma_commit_pair(&c.empty[stage], BOTH_CTAS);
                if (++stage == ring.nst) {
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
        }
    } else if (warp >= 2 && warp < kGatherWarp0) {
        // ------------------------------ epilogue (both CTAs) ------------------------------
        const int quarter = warp & 3;
        const int r_local = quarter * 32 + lane;
        uint32_t acc = 0, acc_phase = 0;
        bool aborted = false;
        for (int i = walk.first; i < walk.count && !aborted; i += walk.stride) {
          const PairItem slot = slot_at(i);
          for (int sub = 0; sub < slot.nsub; ++sub) {
            PairItem it = slot;
            it.n_tile += sub;
            if (!ptx::mbar_wait(&c.tfull[acc], acc_phase, abort_flag)) {
                raise_abort(c, status);
                aborted = true;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * ACC_COLS;
            const bool kfull = it.kslice * kb_per < num_kb;  // an empty K slice contributes zeros
            if (SWAPCAP && it.swap) {
                // Accumulator lane = weight column col0 of this CTA's half, accumulator column = row;
                // the second MMA's accumulator (at +128) holds kind 0's up column / kind 1's column
                // col0 + 256.
                const int col0 = it.n_tile * super_n<KIND>() + 128 * rank + r_local;
                const int nchunk = (it.rows + 31) / 32;
                // FP8: column scales of this lane's two columns (gate/up, or col0/col0+256).
                float sc0 = 1.0f, sc1 = 1.0f;
                if (FP8) {
                    const float* sbe = b_scale + static_cast<size_t>(it.e) * wrows;
                    if (col0 < N) sc0 = __ldg(sbe + col0);
                    if (KIND == 0 ? col0 < N : col0 + 256 < N) sc1 = __ldg(sbe + col0 + (KIND == 0 ? N : 256));
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
                    if (KIND == 1) {
                        float* y = reinterpret_cast<float*>(out) + static_cast<size_t>(it.kslice) * M * N;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nrow) {
                                if (col0 < N) y[(row_base + j) * N + col0] = kfull ? __uint_as_float(a0[j]) : 0.0f;
                                if (col0 + 256 < N)
                                    y[(row_base + j) * N + col0 + 256] = kfull ? __uint_as_float(a1[j]) : 0.0f;
                            }
                    } else if (col0 < N) {
                        {
                            uint16_t* h = reinterpret_cast<uint16_t*>(out);
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j < nrow)
                                    h[(row_base + j) * N + col0] =
                                        bf16_bits(silu_mul(__uint_as_float(a0[j]), __uint_as_float(a1[j])));
                        }
                    }
                }
            } else {
                const int n0 = it.n_tile * BN_OUT;
                const bool row_ok = r_local < it.rows;
                const size_t grow = static_cast<size_t>(it.row0 + r_local);
                // FP8: this lane's row scale and the expert's column scales.
                const float srow = (FP8 && row_ok) ? __ldg(a_scale + grow) : 1.0f;
                const float* sbe = FP8 ? b_scale + static_cast<size_t>(it.e) * wrows : nullptr;
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
                                dst[v] = make_float4(kfull ? __uint_as_float(v32[4 * v]) : 0.0f,
                                                     kfull ? __uint_as_float(v32[4 * v + 1]) : 0.0f,
                                                     kfull ? __uint_as_float(v32[4 * v + 2]) : 0.0f,
                                                     kfull ? __uint_as_float(v32[4 * v + 3]) : 0.0f);
                        }
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
            if (KIND == 1 && fold.cnt != nullptr) {
                // Combine fold (FoldArgs), after the accumulator is released: this thread's y stores
                // are fenced, then its rows' blocks counted.  Normal items: the thread stored all 256
                // columns of its row (four 64-column blocks).  Swapped items: this warp stored the 32
                // columns c0 + 32 q.. and c0 + 256 + 32 q.. (c0 = the CTA's first column, q = its
                // lane quarter) of every row of the chunk, half of two blocks; lane j % 32 counts row j.
                const float* y0 = reinterpret_cast<const float*>(out);
                __threadfence();
                if (SWAPCAP && it.swap) {
                    __syncwarp();
                    const int c0 = it.n_tile * super_n<KIND>() + 128 * rank + 32 * quarter;
                    for (int j = lane; j < it.rows; j += 32) {
                        if (c0 < N) fold_arrive(fold, y0, M, N, ksplit, it.row0 + j, c0 / kFoldCols, 1, status);
                        if (c0 + 256 < N)
                            fold_arrive(fold, y0, M, N, ksplit, it.row0 + j, (c0 + 256) / kFoldCols, 1, status);
                    }
                } else if (r_local < it.rows) {
                    const int n0 = it.n_tile * BN_OUT;
                    for (int q = 0; q < BN_OUT / kFoldCols; ++q)
                        if (n0 + q * kFoldCols < N)
                            fold_arrive(fold, y0, M, N, ksplit, it.row0 + r_local, n0 / kFoldCols + q, kFoldWays, status);
                }
            }
          }
        }
    }

    // ------------------------------ teardown ------------------------------
    if (GATHER && warp >= kGatherWarp0) ptx::cp_async_wait_all();  // no gather copy outlives the CTA
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0 && c.abort_flag) {
        if (leader) {
            // CTA 0's full barriers count both CTAs' copies: wait for every stage filled so far.
            for (int s = 0; s < STAGES_MAX; ++s)
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

template <int KIND, bool SWAPCAP, bool GATHER, bool FP8>
cudaError_t launch_pair_kind(const GemmArgs& a, int num_sms, cudaStream_t s, const char** why) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_2sm_kernel<KIND, SWAPCAP, GATHER, FP8>,
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
    // FP8: activation codes [M, K] and blocked transposed weight codes (one 8 KB block per box).
    const bool maps_ok =
        FP8 ? make_tensor_map_u8(&mA, a.A, a.K, arows, BM) && make_tensor_map_u8(&mA32, a.A, a.K, arows, TOK_BOX_ROWS) &&
                  make_tensor_map_w8(&mB, a.B, a.K, static_cast<uint64_t>(a.E) * bcols, 64)
            : make_tensor_map_bf16(&mA, a.A, a.K, arows, BM) &&
                  make_tensor_map_bf16(&mA32, a.A, a.K, arows, TOK_BOX_ROWS) &&
                  make_tensor_map_bf16(&mB, a.B, bcols, static_cast<uint64_t>(a.E) * a.K, BK);
    if (!maps_ok) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point missing or bad operand)";
        return cudaErrorInvalidValue;
    }
    const int grid = num_sms & ~1;  // whole CTA pairs
    const int ksplit = KIND == 0 ? 1 : a.ksplit;
    const int swap_max = a.pair_swap_max < 0 ? 0 : (a.pair_swap_max > PAIR_SWAP_MAX_ROWS ? PAIR_SWAP_MAX_ROWS
                                                                                      : a.pair_swap_max);
    return launch_k(KIND == 0 ? kPdlGateUp : kPdlDown, grouped_gemm_2sm_kernel<KIND, SWAPCAP, GATHER, FP8>,
                    dim3(grid), dim3(GATHER ? GATHER_THREADS : NUM_THREADS), SMEM_BYTES, s, mA, mA32, mB, a.offsets,
                    a.M, a.K, a.N, a.E, ksplit, swap_max, a.pair_layout, a.pair_split,
                    reinterpret_cast<const int4*>(a.A), a.gather_src, a.gather_T, a.a_scale, a.b_scale, a.out,
                    a.status, a.fold);
}

}  // namespace

cudaError_t launch_grouped_gemm_pair(int kind, const GemmArgs& a, int num_sms, cudaStream_t s,
                                     const char** why) {
    if (a.fp8) {
        if (kind == 1)
            return a.pair == 2 ? launch_pair_kind<1, true, false, true>(a, num_sms, s, why)
                               : launch_pair_kind<1, false, false, true>(a, num_sms, s, why);
        return a.pair == 2 ? launch_pair_kind<0, true, false, true>(a, num_sms, s, why)
                           : launch_pair_kind<0, false, false, true>(a, num_sms, s, why);
    }
    if (kind == 1)
        return a.pair == 2 ? launch_pair_kind<1, true, false, false>(a, num_sms, s, why)
                           : launch_pair_kind<1, false, false, false>(a, num_sms, s, why);
    if (a.gather_src)
        return a.pair == 2 ? launch_pair_kind<0, true, true, false>(a, num_sms, s, why)
                           : launch_pair_kind<0, false, true, false>(a, num_sms, s, why);
    return a.pair == 2 ? launch_pair_kind<0, true, false, false>(a, num_sms, s, why)
                       : launch_pair_kind<0, false, false, false>(a, num_sms, s, why);
}

}  // namespace moe
