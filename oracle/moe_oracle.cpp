// moe_oracle.cpp — plain, slow, CPU reference of one Mixture-of-Experts FFN layer forward.
//
// TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline
// and reference legs may load this library.  The product path (libmoe.so) never calls it, and
// this file shares no code, header, table or helper with the CUDA library.
//
// What the layer computes (the plain definition, step by step):
//   1. route    top-k experts per token from fp32 router logits; weights = softmax over all
//               experts, restricted to the chosen k and renormalised to sum to 1.
//   2. permute  group the (token, slot) assignments by expert (counting sort: expert, then
//               ascending token), giving counts, offsets, src (row -> token), dest (token,slot -> row).
//   3. gate+up  for every permuted row: g = x.W_gate[e], u = x.W_up[e] (fp32 accumulate),
//               h = silu(g) * u, silu(z) = z / (1 + exp(-z)).  h stays fp32 here.
//   4. down     y = h.W_down[e] (fp32 accumulate).
//   5. combine  out[t] = sum_j w[t,j] * y[dest[t,j]], j in slot order, fp32.
//
// Sources:
//   * Stage order dispatch -> linear1 -> SwiGLU -> linear2 -> combine: DeepGEMM PR #304 write-up
//     (itsolotime.com), section 1.1 "the core of the problem: the NVLink bottleneck in MoE inference".
//   * SwiGLU between a fused gate/up projection and the down projection, with the gate/up
//     pre-activations kept out of global memory: "Triton-MoE-Dispatch-Kernel erreicht 131 % von
//     Megablocks" (lumeric.app), the article body.
//   * Rearrange -> GroupGEMM -> weighted-average reduce: the HPC-Ops operator-library page
//     (ntfzh.com), its FusedMoE paragraph.
//   * Top-k routing done on the device inside the MoE kernel: "Triton MoE 核心擊敗 Megablocks"
//     (setupai.cc), section 技術深入 (technical deep dive), the dynamic-routing bullet.
//   The pages never define the router function.  Reading adopted here for every workload:
//   softmax over all E logits, keep the k largest logits (ties -> lower expert index; the slot
//   order is descending logit), renormalise the kept probabilities to sum to 1.
//   A second router, DeepSeek-V3's (the pages only name that model), follows the DeepSeek-V3
//   Technical Report: sigmoid affinities, a selection-only bias, group-limited top-k, normalised
//   and scaled gating values (oracle_route_grouped).
//
// Precision: every floating-point step is fp32 from the same bf16 inputs (bf16 -> fp32 is exact).
// The layer's definition fixes fp32 accumulation; this file is built with -ffp-contract=off so the
// x86 and Arm builds round identically.
//
// Parity pins: every function below is pinned by CPU tests that do not reuse this code
// (tests/test_oracle_pins.py): a hand-worked 4-token example with closed-form outputs, the
// E=1/k=1 dense SwiGLU FFN against numpy matmul, a float64 brute-force per-token dense FFN,
// numpy stable argsort for routing and the permutation, and the layer's invariants.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// bf16 is the upper half of an IEEE fp32 word, so widening is a 16-bit shift (exact).
inline float bf16_to_f32(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return f;
}

inline float silu(float z) { return z / (1.0f + std::exp(-z)); }

// fp32 -> bf16, round to nearest even (finite inputs).
inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return static_cast<uint16_t>(u >> 16);
}

// FP8 E4M3 (the OCP 8-bit floating-point format's E4M3 variant): 1 sign bit, 4 exponent bits
// with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448 = 1.75 * 2^8;
// normals 1.m * 2^(e-7) for e = 1..15 (e = 15 with m = 7 excluded); subnormals m/8 * 2^-6.
inline float e4m3_decode(uint8_t c) {
    const int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return std::nanf("");
    const double v = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
    return static_cast<float>(sgn ? -v : v);
}

// Round to the nearest E4M3 value, ties to even mantissa; magnitudes that round above 448 become
// 448 (saturation to the largest finite value).  NaN maps to the NaN code.
inline uint8_t e4m3_encode(float x) {
    if (std::isnan(x)) return 0x7F;
    const uint8_t sgn = std::signbit(x) ? 0x80 : 0x00;
    const double a = std::fabs(static_cast<double>(x));
    // Quantum of the binade holding a (subnormal range: 2^-9).
    int ex = 0;
    std::frexp(a, &ex);                  // a = f * 2^ex, f in [0.5, 1)
    const int e_unb = a > 0 ? std::max(ex - 1, -6) : -6;  // unbiased exponent, floor at the subnormal one
    const double quantum = std::ldexp(1.0, e_unb - 3);
    const double q = std::nearbyint(a / quantum);  // default rounding mode: to nearest, ties to even
    double v = q * quantum;
    if (v > 448.0) v = 448.0;
    // Encode v (exactly representable by construction).
    if (v == 0.0) return sgn;
    int e2 = 0;
    const double f2 = std::frexp(v, &e2);  // v = f2 * 2^e2
    int exp_field = (e2 - 1) + 7;
    int man;
    if (exp_field <= 0) {  // subnormal: v = m/8 * 2^-6
        exp_field = 0;
        man = static_cast<int>(std::lround(v / std::ldexp(1.0, -9)));
    } else {
        man = static_cast<int>(std::lround((f2 * 2.0 - 1.0) * 8.0));
    }
    return static_cast<uint8_t>(sgn | (exp_field << 3) | man);
}

// Per-row FP8 quantisation of a [R, C] matrix: absmax over the row, inv = 448 / absmax (fp32),
// code = e4m3(value * inv), dequantisation scale = absmax / 448 (fp32); an all-zero row gets
// scale 1 and zero codes.
template <class GetF>
void quantize_rows_fp8(GetF get, int R, int C, uint8_t* q, float* scale) {
    for (int r = 0; r < R; ++r) {
        float amax = 0.0f;
        for (int c = 0; c < C; ++c) amax = std::max(amax, std::fabs(get(r, c)));
        const float inv = amax > 0.0f ? 448.0f / amax : 1.0f;
        scale[r] = amax > 0.0f ? amax / 448.0f : 1.0f;
        for (int c = 0; c < C; ++c) q[static_cast<size_t>(r) * C + c] = e4m3_encode(get(r, c) * inv);
    }
}

// Blockwise FP8 scale of a block with absolute maximum amax: the smallest power of two P with
// fl(amax / 448) <= P (a UE8M0-representable scale), at least 2^-126 so that 1/P is a finite fp32
// power of two; an all-zero block gets P = 1.  Codes are e4m3(v * (1/P)) (exact scaling), the
// dequantised value code * P.
inline float pow2_block_scale(float amax) {
    if (!(amax > 0.0f)) return 1.0f;
    const float q = amax / 448.0f;
    int e = 0;
    const float m = std::frexp(q, &e);  // q = m * 2^e, m in [0.5, 1)
    const float p = (m == 0.5f) ? q : std::ldexp(1.0f, e);
    return std::max(p, std::ldexp(1.0f, -126));
}

// Quantise the C values get(c), c in [0, C), in consecutive blocks of B (C % B == 0): codes q[c],
// one scale per block.
template <class GetF>
void quantize_blocks_fp8(GetF get, int C, int B, uint8_t* q, float* scale) {
    for (int b = 0; b < C / B; ++b) {
        float amax = 0.0f;
        for (int c = b * B; c < (b + 1) * B; ++c) amax = std::max(amax, std::fabs(get(c)));
        const float P = pow2_block_scale(amax);
        const float inv = 1.0f / P;  // exact: P is a power of two in [2^-126, 2^128)
        scale[b] = P;
        for (int c = b * B; c < (b + 1) * B; ++c) q[c] = e4m3_encode(get(c) * inv);
    }
}

// One permuted row through expert e: g, u over i = 0..d-1 ascending; h = silu(g) * u.
void gateup_row(const float* x, const uint16_t* Wgu_e, int d, int f, float* h, float* g, float* u) {
    for (int n = 0; n < f; ++n) { g[n] = 0.0f; u[n] = 0.0f; }
    for (int i = 0; i < d; ++i) {
        const float xi = x[i];
        const uint16_t* wrow = Wgu_e + static_cast<size_t>(i) * 2 * f;   // row i of [d, 2f]
        for (int n = 0; n < f; ++n) {
            g[n] += xi * bf16_to_f32(wrow[n]);          // gate: columns 0 .. f-1
            u[n] += xi * bf16_to_f32(wrow[f + n]);      // up:   columns f .. 2f-1
        }
    }
    for (int n = 0; n < f; ++n) h[n] = silu(g[n]) * u[n];
}

// y = h . W_down[e], n = 0..f-1 ascending.
void down_row(const float* h, const uint16_t* Wd_e, int d, int f, float* y) {
    for (int m = 0; m < d; ++m) y[m] = 0.0f;
    for (int n = 0; n < f; ++n) {
        const float hn = h[n];
        const uint16_t* wrow = Wd_e + static_cast<size_t>(n) * d;       // row n of [f, d]
        for (int m = 0; m < d; ++m) y[m] += hn * bf16_to_f32(wrow[m]);
    }
}

bool valid_shape(int T, int E, int k) { return T >= 0 && E >= 1 && k >= 1 && k <= E; }

}  // namespace

extern "C" {

// Threads OpenMP will use in the parallel loops below.
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

// Step 1, route.  logits [T,E] fp32 row-major -> idx [T,k] int32, w [T,k] fp32.
// Returns 0, or -1 on a bad shape.
int oracle_route(const float* logits, int T, int E, int k, int32_t* idx, float* w) {
    if (!valid_shape(T, E, k)) return -1;
    std::vector<int> order(E);
    std::vector<float> p(E);
    for (int t = 0; t < T; ++t) {
        const float* l = logits + static_cast<size_t>(t) * E;
        // Sort expert ids by logit, largest first; stable, so equal logits keep ascending id.
        // A NaN logit ranks below every number (the NaNs keep ascending id among themselves), which
        // keeps the comparison a strict weak order; the weights of a row with a NaN are undefined.
        std::iota(order.begin(), order.end(), 0);
        std::stable_sort(order.begin(), order.end(), [l](int a, int b) {
            if (std::isnan(l[a])) return false;
            if (std::isnan(l[b])) return true;
            return l[a] > l[b];
        });
        // Full softmax over all E experts.
        float mx = l[0];
        for (int e = 1; e < E; ++e) mx = std::max(mx, l[e]);
        float Z = 0.0f;
        for (int e = 0; e < E; ++e) { p[e] = std::exp(l[e] - mx); Z += p[e]; }
        for (int e = 0; e < E; ++e) p[e] /= Z;
        // Keep the first k in slot order, renormalise.
        float s = 0.0f;
        for (int j = 0; j < k; ++j) s += p[order[j]];
        for (int j = 0; j < k; ++j) {
            idx[static_cast<size_t>(t) * k + j] = order[j];
            w[static_cast<size_t>(t) * k + j] = p[order[j]] / s;
        }
    }
    return 0;
}

// Step 1, second router: DeepSeek-V3's sigmoid gating with a selection bias and group-limited
// top-k (DeepSeek-V3 Technical Report, section 2.1.2: the affinity s = sigmoid(logit); the bias b
// of auxiliary-loss-free load balancing enters only the choice of experts; the gating values are
// the chosen experts' s normalised to sum to 1; the node-limited routing paragraph: experts are
// split into groups and a token may use only the groups with the largest sums of their K_r/M
// highest scores).  Per token, in fp32:
//   s[e] = 1 / (1 + exp(-logit[e]))              affinity
//   c[e] = s[e] + bias[e]                        selection score
//   group g = experts [g*E/G, (g+1)*E/G); its score = sum of its q largest c, q = max(1, k/topk_group)
//   keep the topk_group groups with the largest scores (equal scores -> lower group id)
//   idx = the k experts of the kept groups with the largest c (equal -> lower id), slot order =
//         descending c
//   w[j] = scale * s[idx[j]] / sum_j' s[idx[j']]
// Returns 0, or -1 on a bad shape (E % G != 0, topk_group outside [1, G], k > topk_group * E / G).
int oracle_route_grouped(const float* logits, const float* bias, int T, int E, int k, int n_group,
                         int topk_group, float scale, int32_t* idx, float* w) {
    if (!valid_shape(T, E, k) || n_group < 1 || E % n_group != 0 || topk_group < 1 ||
        topk_group > n_group || k > topk_group * (E / n_group))
        return -1;
    const int gs = E / n_group;
    const int q = std::min(gs, std::max(1, k / topk_group));
    std::vector<float> sc(E), c(E), gscore(n_group), tmp(gs);
    std::vector<int> gorder(n_group), eorder;
    std::vector<char> kept(n_group);
    for (int t = 0; t < T; ++t) {
        const float* l = logits + static_cast<size_t>(t) * E;
        for (int e = 0; e < E; ++e) {
            sc[e] = 1.0f / (1.0f + std::exp(-l[e]));
            c[e] = sc[e] + bias[e];
        }
        // Group scores: the q largest selection scores of each group, added largest first.
        for (int g = 0; g < n_group; ++g) {
            for (int i = 0; i < gs; ++i) tmp[i] = c[g * gs + i];
            std::sort(tmp.begin(), tmp.end(), [](float a, float b) { return a > b; });
            float sum = 0.0f;
            for (int i = 0; i < q; ++i) sum += tmp[i];
            gscore[g] = sum;
        }
        std::iota(gorder.begin(), gorder.end(), 0);
        std::stable_sort(gorder.begin(), gorder.end(), [&](int a, int b) { return gscore[a] > gscore[b]; });
        std::fill(kept.begin(), kept.end(), 0);
        for (int i = 0; i < topk_group; ++i) kept[gorder[i]] = 1;
        // Candidates: the kept groups' experts, ascending id; a stable sort by c keeps equal
        // scores in ascending id.
        eorder.clear();
        for (int e = 0; e < E; ++e)
            if (kept[e / gs]) eorder.push_back(e);
        std::stable_sort(eorder.begin(), eorder.end(), [&](int a, int b) { return c[a] > c[b]; });
        float ssum = 0.0f;
        for (int j = 0; j < k; ++j) ssum += sc[eorder[j]];
        for (int j = 0; j < k; ++j) {
            idx[static_cast<size_t>(t) * k + j] = eorder[j];
            w[static_cast<size_t>(t) * k + j] = scale * (sc[eorder[j]] / ssum);
        }
    }
    return 0;
}

// Step 2, permute: counting sort of the T*k assignments by expert, tokens ascending within an
// expert.  counts [E], offsets [E+1] (exclusive scan), src [T*k] (row -> token),
// dest [T,k] ((token, slot) -> row).  Returns 0, -1 on a bad shape, -2 if idx holds an id
// outside [0,E) or repeats an expert within one token.
int oracle_permute(const int32_t* idx, int T, int E, int k,
                   int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dest) {
    if (!valid_shape(T, E, k)) return -1;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            const int e = idx[static_cast<size_t>(t) * k + j];
            if (e < 0 || e >= E) return -2;
            for (int jj = 0; jj < j; ++jj)
                if (idx[static_cast<size_t>(t) * k + jj] == e) return -2;
        }
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (size_t a = 0; a < static_cast<size_t>(T) * k; ++a) counts[idx[a]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    std::vector<int32_t> cursor(offsets, offsets + E);
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            const int e = idx[static_cast<size_t>(t) * k + j];
            const int r = cursor[e]++;
            src[r] = t;
            dest[static_cast<size_t>(t) * k + j] = r;
        }
    return 0;
}

// x_perm[r] = x[src[r]] for r < M (a bf16 row copy).
void oracle_gather_rows(const uint16_t* x, const int32_t* src, int M, int d, uint16_t* x_perm) {
    for (int r = 0; r < M; ++r)
        std::memcpy(x_perm + static_cast<size_t>(r) * d, x + static_cast<size_t>(src[r]) * d,
                    sizeof(uint16_t) * d);
}

// Step 3, gate+up with SwiGLU over the permuted rows 0..offsets[E]-1 of x_perm [M,d] bf16.
// W_gate_up [E, d, 2f] bf16 (gate columns 0..f-1, up columns f..2f-1) -> h [M, f] fp32.
void oracle_gateup_swiglu(const uint16_t* x_perm, const int32_t* offsets, int E,
                          const uint16_t* Wgu, int d, int f, float* h) {
    for (int e = 0; e < E; ++e) {
        const uint16_t* We = Wgu + static_cast<size_t>(e) * d * 2 * f;
#pragma omp parallel
        {
            std::vector<float> x(d), g(f), u(f);
#pragma omp for schedule(dynamic, 1)
            for (int r = offsets[e]; r < offsets[e + 1]; ++r) {
                for (int i = 0; i < d; ++i) x[i] = bf16_to_f32(x_perm[static_cast<size_t>(r) * d + i]);
                gateup_row(x.data(), We, d, f, h + static_cast<size_t>(r) * f, g.data(), u.data());
            }
        }
    }
}

// Step 4, down projection over rows 0..offsets[E]-1: y [M, d] = h [M, f] . W_down[e] [f, d].
void oracle_down(const float* h, const int32_t* offsets, int E, const uint16_t* Wd, int d, int f,
                 float* y) {
    for (int e = 0; e < E; ++e) {
        const uint16_t* We = Wd + static_cast<size_t>(e) * f * d;
#pragma omp parallel for schedule(dynamic, 1)
        for (int r = offsets[e]; r < offsets[e + 1]; ++r)
            down_row(h + static_cast<size_t>(r) * f, We, d, f, y + static_cast<size_t>(r) * d);
    }
}

// Step 4 with a bf16 h operand (for checking the down-projection stage on its own).
void oracle_down_bf16(const uint16_t* h_bf16, const int32_t* offsets, int E, const uint16_t* Wd,
                      int d, int f, float* y) {
    for (int e = 0; e < E; ++e) {
        const uint16_t* We = Wd + static_cast<size_t>(e) * f * d;
#pragma omp parallel
        {
            std::vector<float> h(f);
#pragma omp for schedule(dynamic, 1)
            for (int r = offsets[e]; r < offsets[e + 1]; ++r) {
                for (int n = 0; n < f; ++n) h[n] = bf16_to_f32(h_bf16[static_cast<size_t>(r) * f + n]);
                down_row(h.data(), We, d, f, y + static_cast<size_t>(r) * d);
            }
        }
    }
}

// Step 5, combine: out[t] = sum over slots j = 0..k-1 (ascending) of w[t,j] * y[dest[t,j]].
void oracle_combine(const float* y, const float* w, const int32_t* dest, int T, int d, int k,
                    float* out) {
#pragma omp parallel for
    for (int t = 0; t < T; ++t) {
        float* o = out + static_cast<size_t>(t) * d;
        for (int m = 0; m < d; ++m) o[m] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const float wj = w[static_cast<size_t>(t) * k + j];
            const float* yr = y + static_cast<size_t>(dest[static_cast<size_t>(t) * k + j]) * d;
            for (int m = 0; m < d; ++m) o[m] += wj * yr[m];
        }
    }
}

// Steps 2-5 for a given routing: idx/w [T,k] (from either router) -> out [T,d] fp32.  x [T,d] bf16,
// W_gate_up [E,d,2f] bf16, W_down [E,f,d] bf16.  Returns 0 or a negative code from permute.
int oracle_forward_routed(const uint16_t* x, const int32_t* idx, const float* w, const uint16_t* Wgu,
                          const uint16_t* Wd, int T, int d, int f, int E, int k, float* out) {
    if (!valid_shape(T, E, k) || d < 1 || f < 1) return -1;
    const size_t M = static_cast<size_t>(T) * k;
    std::vector<int32_t> counts(E), offsets(E + 1), src(M), dest(M);
    int rc = oracle_permute(idx, T, E, k, counts.data(), offsets.data(), src.data(), dest.data());
    if (rc) return rc;
    std::vector<uint16_t> x_perm(M * d);
    oracle_gather_rows(x, src.data(), static_cast<int>(M), d, x_perm.data());
    std::vector<float> h(M * f), y(M * d);
    oracle_gateup_swiglu(x_perm.data(), offsets.data(), E, Wgu, d, f, h.data());
    oracle_down(h.data(), offsets.data(), E, Wd, d, f, y.data());
    oracle_combine(y.data(), w, dest.data(), T, d, k, out);
    return 0;
}

// The whole layer: steps 1-5 in order, with the softmax top-k router.  x [T,d] bf16, logits [T,E]
// fp32, W_gate_up [E,d,2f] bf16, W_down [E,f,d] bf16 -> out [T,d] fp32.  Returns 0 or a negative
// code from route/permute.
int oracle_forward(const uint16_t* x, const float* logits, const uint16_t* Wgu, const uint16_t* Wd,
                   int T, int d, int f, int E, int k, float* out) {
    if (!valid_shape(T, E, k) || d < 1 || f < 1) return -1;
    const size_t M = static_cast<size_t>(T) * k;
    std::vector<int32_t> idx(M);
    std::vector<float> w(M);
    int rc = oracle_route(logits, T, E, k, idx.data(), w.data());
    if (rc) return rc;
    return oracle_forward_routed(x, idx.data(), w.data(), Wgu, Wd, T, d, f, E, k, out);
}

// The layer's output for a chosen subset of tokens only (out_rows [ntok, d] fp32), given those
// tokens' routing idx_rows/w_rows [ntok, k].  Every token's output depends only on its own routing
// and x row, so this is the same definition restricted to those tokens: run each chosen expert's
// FFN on the token's x row, combine in slot order.  Returns 0 or a negative code.
int oracle_forward_tokens_routed(const uint16_t* x, const int32_t* idx_rows, const float* w_rows,
                                 const uint16_t* Wgu, const uint16_t* Wd, int T, int d, int f, int E,
                                 int k, const int32_t* tokens, int ntok, float* out_rows) {
    if (!valid_shape(T, E, k) || d < 1 || f < 1) return -1;
    for (int s = 0; s < ntok; ++s)
        if (tokens[s] < 0 || tokens[s] >= T) return -1;
    const size_t npairs = static_cast<size_t>(ntok) * k;
    for (size_t q = 0; q < npairs; ++q)
        if (idx_rows[q] < 0 || idx_rows[q] >= E) return -2;
    std::vector<float> ys(npairs * d);
#pragma omp parallel
    {
        std::vector<float> xr(d), g(f), u(f), h(f);
#pragma omp for schedule(dynamic, 1)
        for (long long q = 0; q < static_cast<long long>(npairs); ++q) {
            const int s = static_cast<int>(q / k);
            const int e = idx_rows[q];
            const uint16_t* xt = x + static_cast<size_t>(tokens[s]) * d;
            for (int i = 0; i < d; ++i) xr[i] = bf16_to_f32(xt[i]);
            gateup_row(xr.data(), Wgu + static_cast<size_t>(e) * d * 2 * f, d, f, h.data(), g.data(),
                       u.data());
            down_row(h.data(), Wd + static_cast<size_t>(e) * f * d, d, f, ys.data() + q * d);
        }
    }
    for (int s = 0; s < ntok; ++s) {
        float* o = out_rows + static_cast<size_t>(s) * d;
        for (int m = 0; m < d; ++m) o[m] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const float wj = w_rows[static_cast<size_t>(s) * k + j];
            const float* yr = ys.data() + (static_cast<size_t>(s) * k + j) * d;
            for (int m = 0; m < d; ++m) o[m] += wj * yr[m];
        }
    }
    return 0;
}

// The same with the softmax top-k router: each sampled token is routed from its own logits row.
int oracle_forward_tokens(const uint16_t* x, const float* logits, const uint16_t* Wgu,
                          const uint16_t* Wd, int T, int d, int f, int E, int k,
                          const int32_t* tokens, int ntok, float* out_rows) {
    if (!valid_shape(T, E, k) || d < 1 || f < 1) return -1;
    for (int s = 0; s < ntok; ++s)
        if (tokens[s] < 0 || tokens[s] >= T) return -1;
    const size_t npairs = static_cast<size_t>(ntok) * k;
    std::vector<int32_t> idx(npairs);
    std::vector<float> w(npairs);
    for (int s = 0; s < ntok; ++s)
        oracle_route(logits + static_cast<size_t>(tokens[s]) * E, 1, E, k, idx.data() + s * k,
                     w.data() + s * k);
    return oracle_forward_tokens_routed(x, idx.data(), w.data(), Wgu, Wd, T, d, f, E, k, tokens, ntok,
                                        out_rows);
}

// ---------------------------------------------------------------------------------------------
// FP8 variant of the layer (the grouped GEMMs on E4M3 operands).  Scaling: per token for the
// activations (x and h rows), per output channel for the weights (for expert e and output column
// n, over the K dimension) — scales that factor out of each dot product, so
//   g[n] = (sum_i dec(x8[t][i]) * dec(Wgu8[e][n][i])) * (sx[t] * sgu[e][n])    (n < f: gate, f.. up)
//   h    = bf16(silu(g) * u), then quantised per row:  h8, sh[r]
//   y[m] = (sum_n dec(h8[r][n]) * dec(Wd8[e][m][n])) * (sh[r] * sd[e][m])
//   out  = sum_j w_j * y   (slot order)
// Weights are stored transposed, [E, N, K] (K contiguous).
// ---------------------------------------------------------------------------------------------
}  // extern "C"

namespace {
// One row r of the FP8 gate+up GEMM through expert e: decoded codes xd [d] with row scale sx;
// for each of the 2f output columns n (gate n < f, then up), the K sum in ascending i, then the
// product with (sx * se[n]); h = bf16(silu(g) * u).
void gateup_row_fp8(const float* xd, float sx, const uint8_t* We8, const float* se, int d, int f, float* g,
                    float* u, uint16_t* hb) {
    for (int n = 0; n < 2 * f; ++n) {
        const uint8_t* wrow = We8 + static_cast<size_t>(n) * d;
        float acc = 0.0f;
        for (int i = 0; i < d; ++i) acc += xd[i] * e4m3_decode(wrow[i]);
        const float v = acc * (sx * se[n]);
        if (n < f) g[n] = v; else u[n - f] = v;
    }
    for (int n = 0; n < f; ++n) hb[n] = f32_to_bf16_rne(silu(g[n]) * u[n]);
}

// One row of the FP8 down GEMM: decoded h codes hd [f] with row scale sh -> yr [d].
void down_row_fp8(const float* hd, float sh, const uint8_t* Wde8, const float* sde, int d, int f, float* yr) {
    for (int m = 0; m < d; ++m) {
        const uint8_t* wrow = Wde8 + static_cast<size_t>(m) * f;
        float acc = 0.0f;
        for (int n = 0; n < f; ++n) acc += hd[n] * e4m3_decode(wrow[n]);
        yr[m] = acc * (sh * sde[m]);
    }
}
// Blockwise FP8 (128-wide K blocks): one row r through expert e.  xd [d] decoded codes with block
// scales sx[d/128]; weight codes We8 [2f, d] with block scales se[(2f/128) x (d/128)] (row-major by
// output block).  For each output column n the 128-element partial sums are taken block by block
// (i ascending), each multiplied by (sx[b] * se[n/128][b]) and added in block order.
void gateup_row_fp8b(const float* xd, const float* sx, const uint8_t* We8, const float* se, int d, int f,
                     float* g, float* u, uint16_t* hb) {
    const int nb = d / 128;
    for (int n = 0; n < 2 * f; ++n) {
        const uint8_t* wrow = We8 + static_cast<size_t>(n) * d;
        float acc = 0.0f;
        for (int b = 0; b < nb; ++b) {
            float part = 0.0f;
            for (int i = b * 128; i < (b + 1) * 128; ++i) part += xd[i] * e4m3_decode(wrow[i]);
            acc += part * (sx[b] * se[static_cast<size_t>(n / 128) * nb + b]);
        }
        if (n < f) g[n] = acc; else u[n - f] = acc;
    }
    for (int n = 0; n < f; ++n) hb[n] = f32_to_bf16_rne(silu(g[n]) * u[n]);
}

void down_row_fp8b(const float* hd, const float* sh, const uint8_t* Wde8, const float* sde, int d, int f,
                   float* yr) {
    const int nb = f / 128;
    for (int m = 0; m < d; ++m) {
        const uint8_t* wrow = Wde8 + static_cast<size_t>(m) * f;
        float acc = 0.0f;
        for (int b = 0; b < nb; ++b) {
            float part = 0.0f;
            for (int n = b * 128; n < (b + 1) * 128; ++n) part += hd[n] * e4m3_decode(wrow[n]);
            acc += part * (sh[b] * sde[static_cast<size_t>(m / 128) * nb + b]);
        }
        yr[m] = acc;
    }
}
}  // namespace

extern "C" {

uint8_t oracle_e4m3_encode(float x) { return e4m3_encode(x); }
float oracle_e4m3_decode(uint8_t c) { return e4m3_decode(c); }

void oracle_e4m3_encode_array(const float* x, int n, uint8_t* out) {
    for (int i = 0; i < n; ++i) out[i] = e4m3_encode(x[i]);
}
void oracle_e4m3_decode_array(const uint8_t* c, int n, float* out) {
    for (int i = 0; i < n; ++i) out[i] = e4m3_decode(c[i]);
}

// Rows of a bf16 matrix [R, C] -> codes [R, C] and scales [R] (see quantize_rows_fp8).
void oracle_quantize_rows_fp8(const uint16_t* a, int R, int C, uint8_t* q, float* scale) {
    quantize_rows_fp8([&](int r, int c) { return bf16_to_f32(a[static_cast<size_t>(r) * C + c]); }, R, C, q,
                      scale);
}

// Weights W [E, K, N] bf16 -> Wq [E, N, K] codes (transposed) and scales [E, N]: output column n
// of expert e is quantised over its K values like a row.
void oracle_quantize_weights_fp8(const uint16_t* W, int E, int K, int N, uint8_t* Wq, float* scale) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int e = 0; e < E; ++e) {
        const uint16_t* We = W + static_cast<size_t>(e) * K * N;
        quantize_rows_fp8([&](int n, int k) { return bf16_to_f32(We[static_cast<size_t>(k) * N + n]); }, N, K,
                          Wq + static_cast<size_t>(e) * N * K, scale + static_cast<size_t>(e) * N);
    }
}

// The FP8 layer's output for the given tokens (all T of them for the whole layer) with their
// routing idx_rows/w_rows [ntok, k]; out_rows [ntok, d] fp32.  Returns 0 or a negative code.
int oracle_forward_fp8_tokens_routed(const uint16_t* x, const int32_t* idx_rows, const float* w_rows,
                                     const uint8_t* Wgu8, const float* sgu, const uint8_t* Wd8, const float* sd,
                                     int T, int d, int f, int E, int k, const int32_t* tokens, int ntok,
                                     float* out_rows) {
    if (!valid_shape(T, E, k) || d < 1 || f < 1) return -1;
    for (int s = 0; s < ntok; ++s)
        if (tokens[s] < 0 || tokens[s] >= T) return -1;
    const size_t npairs = static_cast<size_t>(ntok) * k;
    for (size_t q = 0; q < npairs; ++q)
        if (idx_rows[q] < 0 || idx_rows[q] >= E) return -2;
    std::vector<float> ys(npairs * d);
#pragma omp parallel
    {
        std::vector<uint8_t> x8(d), h8(f);
        std::vector<float> xd(d), g(f), u(f), hd(f);
        std::vector<uint16_t> hb(f);
        float sx = 0.0f, sh = 0.0f;
#pragma omp for schedule(dynamic, 1)
        for (long long q = 0; q < static_cast<long long>(npairs); ++q) {
            const int s = static_cast<int>(q / k);
            const int e = idx_rows[q];
            oracle_quantize_rows_fp8(x + static_cast<size_t>(tokens[s]) * d, 1, d, x8.data(), &sx);
            for (int i = 0; i < d; ++i) xd[i] = e4m3_decode(x8[i]);
            gateup_row_fp8(xd.data(), sx, Wgu8 + static_cast<size_t>(e) * 2 * f * d, sgu + static_cast<size_t>(e) * 2 * f,
                           d, f, g.data(), u.data(), hb.data());
            oracle_quantize_rows_fp8(hb.data(), 1, f, h8.data(), &sh);
            for (int n = 0; n < f; ++n) hd[n] = e4m3_decode(h8[n]);
            down_row_fp8(hd.data(), sh, Wd8 + static_cast<size_t>(e) * d * f, sd + static_cast<size_t>(e) * d, d, f,
                         ys.data() + q * d);
        }
    }
    for (int s = 0; s < ntok; ++s) {
        float* o = out_rows + static_cast<size_t>(s) * d;
        for (int m = 0; m < d; ++m) o[m] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const float wj = w_rows[static_cast<size_t>(s) * k + j];
            const float* yr = ys.data() + (static_cast<size_t>(s) * k + j) * d;
            for (int m = 0; m < d; ++m) o[m] += wj * yr[m];
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------------------------
// Blockwise FP8 variant: 1 x 128 blocks for the activations (x and h rows), 128 x 128 blocks
// (128 output columns x 128 K values) for the weights, power-of-two block scales (see
// pow2_block_scale).  Per output element, the 128-wide partial sums are scaled block by block:
//   g[n] = sum_b (sum_{i in b} dec(x8[i]) * dec(W8[e][n][i])) * (sx[b] * sw[e][n/128][b])
// ---------------------------------------------------------------------------------------------
float oracle_pow2_block_scale(float amax) { return pow2_block_scale(amax); }

// Rows of a bf16 matrix [R, C] (C % 128 == 0) -> codes [R, C] and scales [R, C/128].
void oracle_quantize_rows_fp8b(const uint16_t* a, int R, int C, uint8_t* q, float* scale) {
    for (int r = 0; r < R; ++r) {
        const uint16_t* row = a + static_cast<size_t>(r) * C;
        quantize_blocks_fp8([&](int c) { return bf16_to_f32(row[c]); }, C, 128, q + static_cast<size_t>(r) * C,
                            scale + static_cast<size_t>(r) * (C / 128));
    }
}

// Weights W [E, K, N] bf16 (K, N multiples of 128) -> codes Wq [E, N, K] (transposed) and scales
// [E, N/128, K/128], one per 128 x 128 block of (output column, K).
void oracle_quantize_weights_fp8b(const uint16_t* W, int E, int K, int N, uint8_t* Wq, float* scale) {
    const int nbn = N / 128, nbk = K / 128;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int e = 0; e < E; ++e)
        for (int bn = 0; bn < nbn; ++bn) {
            const uint16_t* We = W + static_cast<size_t>(e) * K * N;
            for (int bk = 0; bk < nbk; ++bk) {
                float amax = 0.0f;
                for (int n = bn * 128; n < (bn + 1) * 128; ++n)
                    for (int k = bk * 128; k < (bk + 1) * 128; ++k)
                        amax = std::max(amax, std::fabs(bf16_to_f32(We[static_cast<size_t>(k) * N + n])));
                const float P = pow2_block_scale(amax);
                const float inv = 1.0f / P;
                scale[(static_cast<size_t>(e) * nbn + bn) * nbk + bk] = P;
                for (int n = bn * 128; n < (bn + 1) * 128; ++n)
                    for (int k = bk * 128; k < (bk + 1) * 128; ++k)
                        Wq[(static_cast<size_t>(e) * N + n) * K + k] =
                            e4m3_encode(bf16_to_f32(We[static_cast<size_t>(k) * N + n]) * inv);
            }
        }
}

// The blockwise FP8 layer's output for the given tokens with their routing (as
// oracle_forward_fp8_tokens_routed): x rows quantised in 1 x 128 blocks, h likewise.
int oracle_forward_fp8b_tokens_routed(const uint16_t* x, const int32_t* idx_rows, const float* w_rows,
                                      const uint8_t* Wgu8, const float* sgu, const uint8_t* Wd8, const float* sd,
                                      int T, int d, int f, int E, int k, const int32_t* tokens, int ntok,
                                      float* out_rows) {
    if (!valid_shape(T, E, k) || d < 128 || f < 128 || d % 128 || f % 128) return -1;
    for (int s = 0; s < ntok; ++s)
        if (tokens[s] < 0 || tokens[s] >= T) return -1;
    const size_t npairs = static_cast<size_t>(ntok) * k;
    for (size_t q = 0; q < npairs; ++q)
        if (idx_rows[q] < 0 || idx_rows[q] >= E) return -2;
    std::vector<float> ys(npairs * d);
#pragma omp parallel
    {
        std::vector<uint8_t> x8(d), h8(f);
        std::vector<float> xd(d), g(f), u(f), hd(f), sx(d / 128), sh(f / 128);
        std::vector<uint16_t> hb(f);
#pragma omp for schedule(dynamic, 1)
        for (long long q = 0; q < static_cast<long long>(npairs); ++q) {
            const int s = static_cast<int>(q / k);
            const int e = idx_rows[q];
            oracle_quantize_rows_fp8b(x + static_cast<size_t>(tokens[s]) * d, 1, d, x8.data(), sx.data());
            for (int i = 0; i < d; ++i) xd[i] = e4m3_decode(x8[i]);
            gateup_row_fp8b(xd.data(), sx.data(), Wgu8 + static_cast<size_t>(e) * 2 * f * d,
                            sgu + static_cast<size_t>(e) * (2 * f / 128) * (d / 128), d, f, g.data(), u.data(),
                            hb.data());
            oracle_quantize_rows_fp8b(hb.data(), 1, f, h8.data(), sh.data());
            for (int n = 0; n < f; ++n) hd[n] = e4m3_decode(h8[n]);
            down_row_fp8b(hd.data(), sh.data(), Wd8 + static_cast<size_t>(e) * d * f,
                          sd + static_cast<size_t>(e) * (d / 128) * (f / 128), d, f, ys.data() + q * d);
        }
    }
    for (int s = 0; s < ntok; ++s) {
        float* o = out_rows + static_cast<size_t>(s) * d;
        for (int m = 0; m < d; ++m) o[m] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const float wj = w_rows[static_cast<size_t>(s) * k + j];
            const float* yr = ys.data() + (static_cast<size_t>(s) * k + j) * d;
            for (int m = 0; m < d; ++m) o[m] += wj * yr[m];
        }
    }
    return 0;
}

// Blockwise FP8 steps 3 and 4 on their own (as oracle_gateup_swiglu_fp8 / oracle_down_fp8), with
// block scales sx [M, d/128], sgu [E, 2f/128, d/128], sh [M, f/128], sd [E, d/128, f/128].
void oracle_gateup_swiglu_fp8b(const uint8_t* x8_perm, const float* sx, const int32_t* offsets, int E,
                               const uint8_t* Wgu8, const float* sgu, int d, int f, uint16_t* h) {
    for (int e = 0; e < E; ++e) {
#pragma omp parallel
        {
            std::vector<float> xd(d), g(f), u(f);
#pragma omp for schedule(dynamic, 1)
            for (int r = offsets[e]; r < offsets[e + 1]; ++r) {
                for (int i = 0; i < d; ++i) xd[i] = e4m3_decode(x8_perm[static_cast<size_t>(r) * d + i]);
                gateup_row_fp8b(xd.data(), sx + static_cast<size_t>(r) * (d / 128),
                                Wgu8 + static_cast<size_t>(e) * 2 * f * d,
                                sgu + static_cast<size_t>(e) * (2 * f / 128) * (d / 128), d, f, g.data(), u.data(),
                                h + static_cast<size_t>(r) * f);
            }
        }
    }
}

void oracle_down_fp8b(const uint8_t* h8, const float* sh, const int32_t* offsets, int E, const uint8_t* Wd8,
                      const float* sd, int d, int f, float* y) {
    for (int e = 0; e < E; ++e) {
#pragma omp parallel
        {
            std::vector<float> hd(f);
#pragma omp for schedule(dynamic, 1)
            for (int r = offsets[e]; r < offsets[e + 1]; ++r) {
                for (int n = 0; n < f; ++n) hd[n] = e4m3_decode(h8[static_cast<size_t>(r) * f + n]);
                down_row_fp8b(hd.data(), sh + static_cast<size_t>(r) * (f / 128), Wd8 + static_cast<size_t>(e) * d * f,
                              sd + static_cast<size_t>(e) * (d / 128) * (f / 128), d, f, y + static_cast<size_t>(r) * d);
            }
        }
    }
}

// Step 3 of the FP8 layer on its own, over rows 0..offsets[E]-1 of a grouped operand:
// x8_perm [M, d] codes with sx [M], Wgu8 [E, 2f, d] with sgu [E, 2f] -> h [M, f] bf16.
void oracle_gateup_swiglu_fp8(const uint8_t* x8_perm, const float* sx, const int32_t* offsets, int E,
                              const uint8_t* Wgu8, const float* sgu, int d, int f, uint16_t* h) {
    for (int e = 0; e < E; ++e) {
#pragma omp parallel
        {
            std::vector<float> xd(d), g(f), u(f);
#pragma omp for schedule(dynamic, 1)
            for (int r = offsets[e]; r < offsets[e + 1]; ++r) {
                for (int i = 0; i < d; ++i) xd[i] = e4m3_decode(x8_perm[static_cast<size_t>(r) * d + i]);
                gateup_row_fp8(xd.data(), sx[r], Wgu8 + static_cast<size_t>(e) * 2 * f * d,
                               sgu + static_cast<size_t>(e) * 2 * f, d, f, g.data(), u.data(),
                               h + static_cast<size_t>(r) * f);
            }
        }
    }
}

// Step 4 of the FP8 layer on its own: h8 [M, f] codes with sh [M], Wd8 [E, d, f] with sd [E, d]
// -> y [M, d] fp32.
void oracle_down_fp8(const uint8_t* h8, const float* sh, const int32_t* offsets, int E, const uint8_t* Wd8,
                     const float* sd, int d, int f, float* y) {
    for (int e = 0; e < E; ++e) {
#pragma omp parallel
        {
            std::vector<float> hd(f);
#pragma omp for schedule(dynamic, 1)
            for (int r = offsets[e]; r < offsets[e + 1]; ++r) {
                for (int n = 0; n < f; ++n) hd[n] = e4m3_decode(h8[static_cast<size_t>(r) * f + n]);
                down_row_fp8(hd.data(), sh[r], Wd8 + static_cast<size_t>(e) * d * f, sd + static_cast<size_t>(e) * d,
                             d, f, y + static_cast<size_t>(r) * d);
            }
        }
    }
}

}  // extern "C"
