/* moe.h — C ABI of libmoe.so: the forward pass of one Mixture-of-Experts FFN layer on a GB300
 * (sm_103a).
 *
 * The layer, in five stream-ordered steps (each a stage call below; moe_forward runs them as four
 * or five launches, see moe_forward_launch_count):
 *   route    -> top-k experts and their weights per token
 *   permute  -> group the (token, slot) assignments by expert, copy x rows into that order
 *   gate+up  -> grouped BF16 GEMM x_perm . [W_gate | W_up] per expert, SwiGLU fused in the
 *               epilogue, so the gate/up pre-activations never reach global memory
 *   down     -> grouped BF16 GEMM h . W_down per expert
 *   combine  -> out[t] = sum_j w[t,j] * y_perm[dest[t,j]]
 * Stage order: DeepGEMM PR #304 write-up (itsolotime.com), section 1.1 (dispatch -> linear1 ->
 * SwiGLU -> linear2 -> combine) and the HPC-Ops page (ntfzh.com), FusedMoE paragraph
 * (rearrange -> GroupGEMM -> weighted-average reduce).  Gate+up fusion with SwiGLU kept on chip:
 * "Triton-MoE-Dispatch-Kernel erreicht 131 % von Megablocks" (lumeric.app), article body.
 *
 * Conventions for every call
 *   - Tensors are row-major and contiguous.  "bf16" buffers hold IEEE bfloat16 values
 *     (passed as void*); fp32 buffers are float; index buffers are int32_t.
 *   - Unless a parameter says "host", every pointer is a DEVICE pointer (cudaMalloc, or a torch
 *     CUDA tensor's data_ptr()) owned by the caller.  The library allocates no device memory,
 *     never frees anything and keeps no pointer after a call returns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls enqueue work on it
 *     and return without synchronising, except moe_get_device_error, which reads back.
 *   - Return value: MOE_OK (0) or a negative MOE_ERR_* code, and moe_last_error_string() (per
 *     calling thread) says why.  On an argument, shape, workspace or device error nothing is
 *     launched; a *_host_batches call whose enqueueing fails at batch b has enqueued the batches
 *     before b.
 *   - Shape limits: 1 <= E <= 256, 1 <= top_k <= min(E, 8), T >= 0 (T = 0 launches nothing),
 *     d and f multiples of 64 in [64, 65536], T * top_k < 2^31 and every buffer < 2^31 rows.
 *   - Only devices of compute capability 10.3 (GB300) are supported: MOE_ERR_UNSUPPORTED else.
 *   - Device-side checks (an expert id outside [0,E), offsets that are not a valid segmentation,
 *     a dest row out of range, a pipeline wait that exceeded its time limit) never fault: the
 *     kernel skips the offending access and ORs a MOE_STATUS_* bit into the caller's status
 *     word, which moe_get_device_error reads.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1) /* null pointer, bad shape or limit */
#define MOE_ERR_UNSUPPORTED (-2) /* not a compute-capability 10.3 device */
#define MOE_ERR_WORKSPACE (-3)   /* workspace missing or smaller than moe_workspace_size() */
#define MOE_ERR_CUDA (-4)        /* a CUDA runtime/driver call or a launch failed */

/* Bits of the device status word (int32). */
#define MOE_STATUS_BAD_EXPERT_ID 0x1 /* permute: an id outside [0,E) or repeated within a token */
#define MOE_STATUS_BAD_OFFSETS 0x2   /* grouped GEMM: offsets not 0 <= ... nondecreasing <= M */
#define MOE_STATUS_BAD_DEST 0x4      /* combine: a dest row outside [0, T*top_k) */
#define MOE_STATUS_WAIT_TIMEOUT 0x8  /* grouped GEMM: a pipeline wait gave up after ~1 s */
#define MOE_STATUS_BAD_SRC 0x10      /* gathering gate+up GEMM or FP8 row quantiser: a src index out of range (row zeroed) */

typedef void* moe_stream_t; /* a cudaStream_t */

/* Bytes of scratch that moe_forward needs for this shape (256-byte aligned pieces: status word,
 * idx, w, counts, offsets, src, dest, x_perm bf16 [T*k,d], h bf16 [T*k,f], y_perm fp32
 * [moe_down_ksplit(), T*k, d], then the combine-fold counters int32 [T, d/64]).
 * Returns 0 for an invalid shape. */
MOE_API size_t moe_workspace_size(int T, int d, int f, int E, int top_k);

/* Byte offsets of moe_forward's intermediates inside the workspace, in this order: status, idx,
 * w, counts, offsets, src, dest, x_perm, h, y_perm, total (11 values written to offsets_out).
 * Lets a caller inspect the intermediates of a moe_forward call.  Returns MOE_OK or
 * MOE_ERR_INVALID_ARG. */
MOE_API int moe_workspace_layout(int T, int d, int f, int E, int top_k, size_t* offsets_out);

/* Step 1 — top-k routing.  Per token t: the top_k largest of logits[t, 0..E-1] (equal logits:
 * lower expert id first) in slot order of descending logit, and w[t,j] = the softmax over all E
 * logits restricted to the chosen experts and renormalised to sum to 1, all in fp32.
 *   logits [T,E] fp32 in;  idx [T,top_k] int32 out;  w [T,top_k] fp32 out.
 * Routing on the device with no host synchronisation: "Triton MoE 核心擊敗 Megablocks"
 * (setupai.cc), section 技術深入, the dynamic-routing bullet.  The pages do not define the
 * router function; softmax-then-top-k-renormalised is the reading used throughout.
 * Weights are defined for finite logits only.  The ids stay well defined for any input: a NaN
 * logit ranks below every number (-inf included), NaNs among themselves by ascending id, so no
 * expert is chosen twice for one token. */
MOE_API int moe_route(const float* logits, int T, int E, int top_k, int32_t* idx, float* w,
              moe_stream_t stream);

/* Step 1, second router — DeepSeek-V3's gating (DeepSeek-V3 Technical Report, section 2.1.2; the
 * pages only name that model, so the definition comes from its report).  Per token, in fp32:
 *   s[e] = 1 / (1 + exp(-logits[t,e]))      affinity
 *   c[e] = s[e] + bias[e]                   selection score (the auxiliary-loss-free balancing bias
 *                                           steers the choice only)
 *   the E experts form n_group equal groups (experts g*E/n_group ..); a group's score is the sum of
 *   its q = max(1, top_k / topk_group) largest c (the report's node-limited routing); the topk_group
 *   best groups are kept (equal scores: lower group first);
 *   idx[t,.] = the top_k largest c among the kept groups' experts (equal: lower id first), in slot
 *   order of descending c;  w[t,j] = scale * s[idx[t,j]] / sum_j' s[idx[t,j']] (sum in slot order).
 *   logits [T,E] fp32 in;  bias [E] fp32 in;  idx [T,top_k] int32 out;  w [T,top_k] fp32 out.
 * DeepSeek-V3's own setting: E = 256, n_group = 8, topk_group = 4, top_k = 8, scale = 2.5.
 * Requires 1 <= n_group <= 32 dividing E, 1 <= topk_group <= n_group, top_k <= topk_group * E /
 * n_group, scale > 0 (else MOE_ERR_INVALID_ARG).  The selection compares fp32 values computed with
 * the GPU's expf: a choice between scores within a few ulp of each other may differ from a CPU
 * evaluation of the same formula; either choice is a valid top-k. */
MOE_API int moe_route_grouped(const float* logits, const float* bias, int T, int E, int top_k, int n_group,
                      int topk_group, float scale, int32_t* idx, float* w, moe_stream_t stream);

/* Step 2 — permute ("dispatch", the data rearrangement before the grouped GEMM).  Groups the
 * T*top_k assignments by expert, tokens ascending within an expert (a stable counting sort, so
 * the result is unique and bit-exact):
 *   idx [T,top_k] int32 in;  x [T,d] bf16 in;
 *   counts [E] int32 out (assignments per expert);  offsets [E+1] int32 out (exclusive scan;
 *   expert e owns rows offsets[e] .. offsets[e+1]-1);  src [T*top_k] int32 out (row -> token);
 *   dest [T,top_k] int32 out ((token, slot) -> row);  x_perm [T*top_k, d] bf16 out (x_perm[r] =
 *   x[src[r]]), or NULL to compute the indices only (for a consumer that gathers or quantises the
 *   rows by src itself);  status: device int32 or NULL, gets MOE_STATUS_BAD_EXPERT_ID.
 * DeepGEMM PR #304 write-up, section 3.1 (m-grouped contiguous layout: activations contiguous by
 * token, grouped per expert); HPC-Ops page, FusedMoE paragraph (the preceding rearrangement). */
MOE_API int moe_permute(const int32_t* idx, const void* x, int T, int d, int E, int top_k,
                int32_t* counts, int32_t* offsets, int32_t* src, int32_t* dest, void* x_perm,
                int32_t* status, moe_stream_t stream);

/* Step 3 — grouped gate+up GEMM with the SwiGLU epilogue.  For every expert e and row r in
 * [offsets[e], offsets[e+1]):  g = x_perm[r] . W_gate_up[e][:, 0:f],  u = x_perm[r] .
 * W_gate_up[e][:, f:2f] (fp32 accumulation on the tensor cores), h[r] = bf16(silu(g) * u),
 * silu(z) = z / (1 + exp(-z)).  g and u live only in tensor memory.
 *   x_perm [M,d] bf16 in;  w_gate_up [E,d,2f] bf16 in;  offsets [E+1] int32 in (device);
 *   M = rows of x_perm and h;  h [M,f] bf16 out (rows past offsets[E] untouched);
 *   status: device int32 or NULL (MOE_STATUS_BAD_OFFSETS, MOE_STATUS_WAIT_TIMEOUT).
 * "Triton-MoE-Dispatch-Kernel erreicht 131 % von Megablocks" (lumeric.app), article body;
 * block-scheduled grouped GEMM over variable expert batches: "Triton MoE 核心擊敗 Megablocks",
 * section 關鍵要點; persistent kernel hiding prologue/epilogue: HPC-Ops page.
 * Experts with at most 64 rows (environment MOE_GEMM_SWAP_MAX overrides; 0 = never) run with
 * A and B swapped — weights as the tensor-core M operand, the expert's rows as N — as in
 * "dynamic swap A/B" of the DeepGEMM PR #304 write-up, section 3.2; results are the same. */
MOE_API int moe_grouped_gemm_gateup_swiglu(const void* x_perm, const void* w_gate_up,
                                   const int32_t* offsets, int M, int d, int f, int E, void* h,
                                   int32_t* status, moe_stream_t stream);

/* Step 3 with the gather fused in: the same operation as moe_grouped_gemm_gateup_swiglu, but row r
 * of the grouped operand is x[src[r]] — the kernel gathers the rows of x itself (16-byte cp.async
 * copies into the tensor-core operand layout), so x_perm never exists in global memory.  moe_forward
 * runs it when the environment sets MOE_GATHER=1 (the permute then only computes the indices); by
 * default it writes x_perm and reads it with TMA, which measured faster.
 *   x [T,d] bf16 in;  src [M] int32 in (row -> token, from moe_permute; an index outside [0, T) is
 *   read as a zero row and sets MOE_STATUS_BAD_SRC);
 *   other arguments as for moe_grouped_gemm_gateup_swiglu.
 * The pages fuse the dispatch steps to cut kernel launches and passes over the activations
 * ("Triton-MoE-Dispatch-Kernel erreicht 131 % von Megablocks", lumeric.app, its bullet list: 24+
 * launches down to 5); folding the row gather into the GEMM removes one more write and read of
 * the T*top_k x d activations. */
MOE_API int moe_grouped_gemm_gateup_swiglu_gather(const void* x, const int32_t* src, int T, const void* w_gate_up,
                                          const int32_t* offsets, int M, int d, int f, int E, void* h,
                                          int32_t* status, moe_stream_t stream);

/* Step 4 — grouped down-projection GEMM: y_perm[r] = h[r] . W_down[e] (fp32 accumulation) for
 * r in expert e's segment.  With ksplit > 1 the reduction over f is split into ksplit contiguous
 * ranges of 64-wide blocks and y_perm receives ksplit partial sums, slice s at y_perm + s*M*d;
 * y_perm[r] is their sum (moe_combine adds them in slice order).  A slice past the end of f holds
 * zeros.
 *   h [M,f] bf16 in;  w_down [E,f,d] bf16 in;  offsets [E+1] int32 in;  ksplit in [1, 8];
 *   y_perm [ksplit, M, d] fp32 out;  status as for step 3.
 * DeepGEMM PR #304 write-up, section 1.1 ("linear2"); HPC-Ops page (GroupGEMM). */
MOE_API int moe_grouped_gemm_down(const void* h, const void* w_down, const int32_t* offsets, int M, int d,
                          int f, int E, int ksplit, float* y_perm, int32_t* status, moe_stream_t stream);

/* Which grouped-GEMM kernel moe_forward (and the stage calls) run for this layer shape, for the
 * gate+up GEMM (kind 0) or the down GEMM (kind 1):
 *   0  single SMs: 128-row tiles, experts with <= 64 rows swapped (weights as the UMMA M operand);
 *   1  SM pairs (tcgen05 cta_group::2), 256-row tiles only;
 *   2  SM pairs that also run small experts, and the short remainders of larger ones, swapped
 *      (M = 256 weight columns x N = rows; up to 64 or 128 rows, by the shared-memory layout the
 *      kernel picks on the device from the row counts);
 *  -1  invalid shape or kind.
 * Policy: with T*top_k >= 128*E (the average expert holds >= 128 rows) SM pairs, mode 2 for
 * gate+up and mode 1 for the down GEMM; from 32 rows per expert, mode 2 for a many-expert layer
 * (E * ceil(f/256) >= 608 for gate+up, E * ceil(d/512) >= 608 for down); else mode 0.
 * The environment variable MOE_GEMM_2SM=0/1/2 overrides both GEMMs, MOE_GEMM_2SM_DOWN the down
 * GEMM alone, MOE_GEMM_PAIR_SWAP_MAX the swap threshold of mode 2 (0..128).  Results agree with
 * the oracle in every mode. */
MOE_API int moe_gemm_pair_mode(int T, int d, int f, int E, int top_k, int kind);

/* The ksplit that moe_forward uses for the down projection of this layer shape (2 when the 1-SM
 * kernel runs and the down projection has between one and two waves of 128x256 work items on a
 * 152-SM GPU, else 1);
 * 0 for an invalid shape.  The environment variable MOE_DOWN_KSPLIT, if set, overrides it. */
MOE_API int moe_down_ksplit(int T, int d, int f, int E, int top_k);

/* Step 5 — weighted combine (unpermute): out[t] = bf16( sum_{j=0..top_k-1} w[t,j] *
 * y_perm[dest[t,j]] ), fp32 sums in slot order; no atomics, so the result is deterministic.
 * y_perm may hold ksplit partial slices from moe_grouped_gemm_down; each row is the sum of its
 * slices, added in slice order.
 *   y_perm [ksplit, T*top_k, d] fp32 in;  w [T,top_k] fp32 in;  dest [T,top_k] int32 in;
 *   ksplit in [1, 8];  out [T,d] bf16 out;  status: device int32 or NULL (MOE_STATUS_BAD_DEST).
 * DeepGEMM PR #304 write-up, section 1.1 ("combine"); HPC-Ops page (weighted-average reduce). */
MOE_API int moe_combine(const float* y_perm, const float* w, const int32_t* dest, int T, int d, int top_k,
                int ksplit, void* out, int32_t* status, moe_stream_t stream);

/* The whole layer in one call: steps 1-5 on `stream` as moe_forward_launch_count() launches,
 * intermediates carved from `workspace` (device, >= moe_workspace_size() bytes, 256-byte aligned).
 * With MOE_FOLD_COMBINE=1 in the environment, step 5 runs inside the down GEMM instead of as its
 * own launch: every (token, 64-column block) has an arrival counter (zeroed by the permute
 * launch); each epilogue that stored its part of a row's block adds its share, and the arrival
 * that completes the token's top_k rows (and K slices) writes that block of `out` — the same fp32
 * sum in slot order as moe_combine, with no atomics on the output, so the result is deterministic
 * and equal to the default form bit for bit.  It is off by default because it is slower: the
 * completing arrival sums top_k rows in one thread, at the tail of the GEMM.
 *   x [T,d] bf16;  logits [T,E] fp32;  w_gate_up [E,d,2f] bf16;  w_down [E,f,d] bf16;
 *   out [T,d] bf16.
 * The status word at the start of the workspace is reset by the first kernel of every call and
 * can be read with moe_get_device_error(workspace, ...) after the stream has run the call. */
MOE_API int moe_forward(const void* x, const float* logits, const void* w_gate_up, const void* w_down,
                int T, int d, int f, int E, int top_k, void* out, void* workspace,
                size_t workspace_bytes, moe_stream_t stream);

/* moe_forward with DeepSeek-V3's router (moe_route_grouped) as step 1; steps 2-5 as in
 * moe_forward, with the same workspace (moe_workspace_size) and five launches (routing and the
 * permutation never fuse with this router; four with MOE_FOLD_COMBINE=1).  bias [E] fp32 and
 * n_group, topk_group, scale as for moe_route_grouped. */
MOE_API int moe_forward_grouped(const void* x, const float* logits, const float* bias, const void* w_gate_up,
                        const void* w_down, int T, int d, int f, int E, int top_k, int n_group,
                        int topk_group, float scale, void* out, void* workspace, size_t workspace_bytes,
                        moe_stream_t stream);

/* moe_forward with the per-call tensors in HOST memory: x_host [T,d] bf16 and logits_host [T,E]
 * fp32 are copied to the device, the layer runs, and out [T,d] bf16 is copied back to out_host,
 * all enqueued on `stream` (cudaMemcpyAsync; page-locked host buffers make the copies
 * asynchronous).  The caller synchronises the stream before reading out_host.  x and logits are
 * staged in the workspace, which must hold moe_workspace_size() + moe_host_staging_size() bytes;
 * out is staged there too.  Weights stay device pointers. */
MOE_API size_t moe_host_staging_size(int T, int d, int E);
MOE_API int moe_forward_host(const void* x_host, const float* logits_host, const void* w_gate_up,
                     const void* w_down, int T, int d, int f, int E, int top_k, void* out_host,
                     void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* moe_forward_host over n_batches batches of T tokens each, with the copies overlapped with the
 * layers: batch i's x [T,d] bf16 and logits [T,E] fp32 are read from x_hosts[i] and
 * logits_hosts[i] and its out [T,d] bf16 is written to out_hosts[i] (page-locked host memory, or
 * the copies do not overlap).  The layers run one after another on `stream`; the host-to-device
 * copies are issued on h2d_stream and the device-to-host copies on d2h_stream (two streams other
 * than `stream`, so that both copy directions run beside the layers), ordered by events: batch
 * i+1's inputs and batch i-1's output move while batch i computes.  Inputs and outputs are staged
 * in two slots after the layer's workspace: workspace_bytes >= moe_workspace_size() +
 * 2 * moe_host_staging_size().  All work is ordered after what `stream` already holds, and
 * `stream` completes only after the last copy back: synchronise `stream` before reading
 * out_hosts.  The call creates seven CUDA events and releases them before returning (the driver
 * frees them once the recorded work completes); it allocates no device memory.  Errors as
 * moe_forward_host; n_batches = 0 does nothing. */
MOE_API int moe_forward_host_batches(const void* const* x_hosts, const float* const* logits_hosts,
                                     const void* w_gate_up, const void* w_down, int n_batches, int T, int d, int f,
                                     int E, int top_k, void* const* out_hosts, void* workspace,
                                     size_t workspace_bytes, moe_stream_t stream, moe_stream_t h2d_stream,
                                     moe_stream_t d2h_stream);

/* moe_forward_host_batches with DeepSeek-V3's router (moe_forward_grouped as the layer): bias [E]
 * fp32 on the device and n_group, topk_group, scale as for moe_route_grouped; the rest as
 * moe_forward_host_batches. */
MOE_API int moe_forward_grouped_host_batches(const void* const* x_hosts, const float* const* logits_hosts,
                                             const float* bias, const void* w_gate_up, const void* w_down,
                                             int n_batches, int T, int d, int f, int E, int top_k, int n_group,
                                             int topk_group, float scale, void* const* out_hosts, void* workspace,
                                             size_t workspace_bytes, moe_stream_t stream, moe_stream_t h2d_stream,
                                             moe_stream_t d2h_stream);

/* Size of the fixed scratch array that moe_forward_noalloc uses (64 MiB). */
#define MOE_NOALLOC_SCRATCH_BYTES (64ull * 1024ull * 1024ull)

/* moe_forward without a caller-provided workspace and without allocating anything.
 * The pages have no counterpart to this call.  It is for callers that cannot allocate device
 * memory at the moment they run the layer: inference servers that carve all device memory into
 * fixed pools at start-up and have none left to hand out, plugins inside a host framework whose
 * allocator they cannot reach, and latency-critical paths where a cudaMalloc (which can
 * synchronise the device) is not acceptable.  Such callers pass only the layer's inputs and output.
 *   x [T,d] bf16, logits [T,E] fp32, w_gate_up [E,d,2f] bf16, w_down [E,f,d] bf16 in;
 *   out [T,d] bf16 out — device pointers, same meaning and layout as moe_forward.
 * The intermediates live in one file-scope device array of MOE_NOALLOC_SCRATCH_BYTES that every
 * GPU loading this library holds until the process exits.  Shapes whose moe_workspace_size()
 * exceeds it are rejected with MOE_ERR_WORKSPACE (e.g. the Mixtral-8x7B shape fits up to
 * T = 628 tokens with top-2).  The first call on a device (and the first after that device's
 * context was destroyed and created again) looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before any stream
 * capture.  Device ordinals >= 64 are rejected with MOE_ERR_UNSUPPORTED.  All calls on a device
 * share the one array and it keeps the last call's contents (every intermediate is rewritten
 * before it is read; the status word is reset by the first kernel), so calls whose work overlaps
 * on the GPU — on different streams, or from different threads without ordering — race with each
 * other: serialise them.  The device status word sits at the start of the array;
 * moe_get_device_error(NULL, &code) reads it for the current device.
 * Returns MOE_OK or an MOE_ERR_* code as moe_forward does. */
MOE_API int moe_forward_noalloc(const void* x, const float* logits, const void* w_gate_up,
                                const void* w_down, int T, int d, int f, int E, int top_k,
                                void* out, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * FP8 (E4M3) variant of the layer.  The grouped GEMMs run on 8-bit E4M3 codes (the OCP FP8
 * format: bias 7, 3 mantissa bits, largest finite 448) on the tensor cores (tcgen05 kind::f8f6f4,
 * fp32 accumulation).  Quantisation: absmax over a row (activations: each x_perm row and each h
 * row) or over an output column's K values (weights), inv = 448 / absmax, code = E4M3(v * inv)
 * rounded to nearest even, saturating at 448; dequantisation scale = absmax / 448 (an all-zero
 * row or column: scale 1, zero codes).  The scales factor out of each dot product, so
 *   g[n] = (sum_i x8[r][i] * W8[e][n][i]) * (sx[r] * s_gate_up[e][n])   (likewise u, y),
 * applied in the GEMM epilogue.  DeepGEMM PR #304 write-up, section 5.3 (an FP8 grouped GEMM on
 * SM100) and its Mega MoE figure (SwiGLU then FP8 quantisation inside the fused layer) are the
 * pages' FP8 context; they scale 128-wide blocks, this variant scales whole rows and columns (its
 * scales then need no per-block promotion of the accumulator).  d and f must be multiples of 128; codes
 * and weight scales 16-byte aligned, row scales 4-byte aligned.
 * ------------------------------------------------------------------------------------------- */

/* Weights, once per model: W [E,K,N] bf16 (as w_gate_up [E,d,2f] or w_down [E,f,d]) -> Wq E4M3
 * codes, transposed and blocked: [E, N/64, K/128, 64, 128], the code of (expert e, output column n,
 * reduction index k) at [e][n/64][k/128][n%64][k%128] — contiguous 8 KB blocks of 64 output
 * columns x 128 K values, which the FP8 GEMMs read as whole blocks — and scale [E,N] fp32, one per
 * output column.  Requires 1 <= E <= 256, K a multiple of 128 and N of 64, both <= 65536. */
MOE_API int moe_quantize_weights_fp8(const void* W, int E, int K, int N, void* Wq, float* scale,
                                     moe_stream_t stream);

/* Step 2 of the FP8 layer: moe_permute, with the permuted rows written as E4M3 codes instead of
 * bf16 — each token's row quantised once (absmax over its d values) and its codes and scale written
 * to each of its top_k rows: x8_perm [T*top_k, d] codes (8-byte aligned), sx [T*top_k] fp32; the
 * other arguments and outputs as for moe_permute. */
MOE_API int moe_permute_fp8(const int32_t* idx, const void* x, int T, int d, int E, int top_k, int32_t* counts,
                            int32_t* offsets, int32_t* src, int32_t* dest, void* x8_perm, float* sx,
                            int32_t* status, moe_stream_t stream);

/* Rows: q[r] = E4M3 codes of row src[r] of a (row r when src is NULL), scale[r] its scale.
 *   a [src_rows, C] bf16 in (16-byte aligned), C a multiple of 8;  src [R] int32 in or NULL (then
 *   src_rows >= R);  q [R, C] codes out (8-byte aligned);  scale [R] fp32 out;
 *   status: device int32 or NULL (a src value outside [0, src_rows) quantises a zero row and sets
 *   MOE_STATUS_BAD_SRC).
 * moe_forward_fp8 uses it on h. */
MOE_API int moe_quantize_rows_fp8(const void* a, const int32_t* src, int R, int C, int src_rows, void* q,
                                  float* scale, int32_t* status, moe_stream_t stream);

/* Step 3 on E4M3 operands: h[r] = bf16(silu(g) * u) with g, u as above.
 *   x8_perm [M,d] codes, sx [M] fp32;  w8_gate_up: blocked codes of the [E,2f,d] transposed
 *   weights (gate columns 0..f-1, up f..2f-1 of each expert), s_gate_up [E,2f] fp32, both from
 *   moe_quantize_weights_fp8 of w_gate_up;
 *   offsets [E+1];  h [M,f] bf16 out;  status as for step 3. */
MOE_API int moe_grouped_gemm_gateup_swiglu_fp8(const void* x8_perm, const float* sx, const void* w8_gate_up,
                                               const float* s_gate_up, const int32_t* offsets, int M, int d,
                                               int f, int E, void* h, int32_t* status, moe_stream_t stream);

/* Step 4 on E4M3 operands: y_perm[r][m] = (sum_n h8[r][n] * W8[e][m][n]) * (sh[r] * s_down[e][m]).
 *   h8 [M,f] codes, sh [M] fp32;  w8_down: blocked codes of the [E,d,f] transposed weights and
 *   s_down [E,d] fp32 (moe_quantize_weights_fp8 of w_down);  ksplit in [1, 8]
 *   (K slices of 128-wide blocks, as in moe_grouped_gemm_down);  y_perm [ksplit,M,d] fp32 out. */
MOE_API int moe_grouped_gemm_down_fp8(const void* h8, const float* sh, const void* w8_down, const float* s_down,
                                      const int32_t* offsets, int M, int d, int f, int E, int ksplit,
                                      float* y_perm, int32_t* status, moe_stream_t stream);

/* The FP8 layer in one call: route (+ permute writing quantised x rows), FP8 gate+up GEMM
 * (+ SwiGLU), quantise h rows, FP8 down GEMM, combine — 5 launches (6 when routing and the
 * permutation run apart; one fewer with MOE_FOLD_COMBINE=1, which folds the combine into the down
 * GEMM as for moe_forward; moe_forward_fp8_launch_count).  Inputs as for moe_forward, with the
 * weights given as moe_quantize_weights_fp8 codes and scales; workspace >=
 * moe_workspace_size_fp8() bytes, 256-byte aligned, its pieces at moe_workspace_layout_fp8()'s
 * offsets: status, idx, w, counts, offsets, src, dest, x8 [M,d], sx [M], h [M,f] bf16, h8 [M,f],
 * sh [M], y_perm [moe_down_ksplit_fp8(), M, d], total (14 values); the combine-fold counters
 * int32 [T, d/64] lie between the end of y_perm and total. */
MOE_API size_t moe_workspace_size_fp8(int T, int d, int f, int E, int top_k);
MOE_API int moe_workspace_layout_fp8(int T, int d, int f, int E, int top_k, size_t* offsets_out);
MOE_API int moe_down_ksplit_fp8(int T, int d, int f, int E, int top_k);
/* As moe_gemm_pair_mode, for moe_forward_fp8's GEMMs.  Policy (the same environment overrides):
 * gate+up as for moe_forward; the down GEMM on normal-only SM pairs (1) from 128 rows per expert on
 * average, else single SMs (0). */
MOE_API int moe_gemm_pair_mode_fp8(int T, int d, int f, int E, int top_k, int kind);
MOE_API int moe_forward_fp8_launch_count(int T, int E, int top_k);
MOE_API int moe_forward_fp8(const void* x, const float* logits, const void* w8_gate_up, const float* s_gate_up,
                            const void* w8_down, const float* s_down, int T, int d, int f, int E, int top_k,
                            void* out, void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Blockwise FP8 variant: the scales vary along K.  Activations (x and h rows) are scaled per
 * 1 x 128 block (one scale per 128 consecutive values of a row), weights per 128 x 128 block of
 * (output column, K).  Block scales are powers of two — the smallest power of two P with
 * fl(absmax / 448) <= P, at least 2^-126, 1 for an all-zero block (representable as UE8M0, the
 * scale encoding of the DeepGEMM write-up's SM100 path, section on the FP4 indexer) — and codes
 * are E4M3(v / P) (exact scaling; round to nearest even, saturating).  The GEMM sums each 128-deep
 * block on the tensor cores and adds block b's partial times (scale_row[b] * scale_col[b]) in block
 * order:  g[n] = sum_b (sum_{i in b} x8[i] * W8[e][n][i]) * (sx[r][b] * sw[e][n/128][b]).
 * "Blockwise FP8" (HPC-Ops page) and the Mega MoE epilogue's FP8 quantisation (DeepGEMM write-up,
 * section 1.2) are the pages' context.  d and f must be multiples of 128; the GEMMs run on single
 * SMs (each 128-deep partial product is promoted into fp32 registers by eight warps).
 * ------------------------------------------------------------------------------------------- */

/* Weights: W [E,K,N] bf16 (K, N multiples of 128) -> Wq blocked codes exactly as
 * moe_quantize_weights_fp8 lays them out, and scale [E, N/128, K/128] fp32 (powers of two).
 * W and Wq 16-byte aligned. */
MOE_API int moe_quantize_weights_fp8b(const void* W, int E, int K, int N, void* Wq, float* scale,
                                      moe_stream_t stream);

/* Rows in 128-wide blocks: q[r] = codes of row src[r] of a (row r when src is NULL), scale [R, C/128].
 * C a multiple of 128; other arguments as for moe_quantize_rows_fp8. */
MOE_API int moe_quantize_rows_fp8b(const void* a, const int32_t* src, int R, int C, int src_rows, void* q,
                                   float* scale, int32_t* status, moe_stream_t stream);

/* Blockwise steps 3 and 4: as moe_grouped_gemm_gateup_swiglu_fp8 / moe_grouped_gemm_down_fp8 with
 * block scales sx [M, d/128], s_gate_up [E, 2f/128, d/128], sh [M, f/128], s_down [E, d/128, f/128]. */
MOE_API int moe_grouped_gemm_gateup_swiglu_fp8b(const void* x8_perm, const float* sx, const void* w8_gate_up,
                                                const float* s_gate_up, const int32_t* offsets, int M, int d,
                                                int f, int E, void* h, int32_t* status, moe_stream_t stream);
/* moe_grouped_gemm_gateup_swiglu_fp8b with h quantised in the GEMM's epilogue, as
 * moe_quantize_rows_fp8b would quantise its bf16 output: h8 [M, f] E4M3 codes (the bf16-rounded
 * h divided by its block's scale) and sh [M, f/128] power-of-two block scales; h in bf16 is never
 * written.  moe_forward_fp8b runs this form.  sh 4-byte aligned; other arguments and errors as the
 * call above. */
MOE_API int moe_grouped_gemm_gateup_swiglu_fp8b_q(const void* x8_perm, const float* sx, const void* w8_gate_up,
                                                  const float* s_gate_up, const int32_t* offsets, int M, int d,
                                                  int f, int E, void* h8, float* sh, int32_t* status,
                                                  moe_stream_t stream);
MOE_API int moe_grouped_gemm_down_fp8b(const void* h8, const float* sh, const void* w8_down, const float* s_down,
                                       const int32_t* offsets, int M, int d, int f, int E, int ksplit,
                                       float* y_perm, int32_t* status, moe_stream_t stream);

/* The blockwise FP8 layer in one call: route (+ permute, indices only), x rows quantised in blocks
 * (gathered by src), blockwise gate+up GEMM (+ SwiGLU), h quantised in blocks, blockwise down GEMM,
 * combine.  When the experts hold more than 64 rows on average (T*top_k > 64*E), h is quantised in
 * the gate+up GEMM's epilogue (moe_grouped_gemm_gateup_swiglu_fp8b_q; h in bf16 is not written),
 * else by its own launch: 5 or 6 launches, one more when routing and the permutation run apart
 * (moe_forward_fp8b_launch_count; moe_fp8b_gemm_quantizes_h tells which form, 1 = in the GEMM,
 * -1 for a bad shape; MOE_FP8B_FUSE_H=0/1 overrides the choice).  Workspace as for
 * moe_forward_fp8 (14 offsets from moe_workspace_layout_fp8b), with sx [T*top_k, d/128] and
 * sh [T*top_k, f/128]. */
MOE_API int moe_fp8b_gemm_quantizes_h(int T, int E, int top_k);
MOE_API size_t moe_workspace_size_fp8b(int T, int d, int f, int E, int top_k);
MOE_API int moe_workspace_layout_fp8b(int T, int d, int f, int E, int top_k, size_t* offsets_out);
MOE_API int moe_down_ksplit_fp8b(int T, int d, int f, int E, int top_k);
MOE_API int moe_forward_fp8b_launch_count(int T, int E, int top_k);
MOE_API int moe_forward_fp8b(const void* x, const float* logits, const void* w8_gate_up, const float* s_gate_up,
                             const void* w8_down, const float* s_down, int T, int d, int f, int E, int top_k,
                             void* out, void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* moe_forward_host_batches with moe_forward_fp8 / moe_forward_fp8b as the layer: the same
 * overlapped copies over two staging slots, weights as those calls take them; workspace_bytes >=
 * moe_workspace_size_fp8() (resp. moe_workspace_size_fp8b()) + 2 * moe_host_staging_size(). */
MOE_API int moe_forward_fp8_host_batches(const void* const* x_hosts, const float* const* logits_hosts,
                                         const void* w8_gate_up, const float* s_gate_up, const void* w8_down,
                                         const float* s_down, int n_batches, int T, int d, int f, int E, int top_k,
                                         void* const* out_hosts, void* workspace, size_t workspace_bytes,
                                         moe_stream_t stream, moe_stream_t h2d_stream, moe_stream_t d2h_stream);
MOE_API int moe_forward_fp8b_host_batches(const void* const* x_hosts, const float* const* logits_hosts,
                                          const void* w8_gate_up, const float* s_gate_up, const void* w8_down,
                                          const float* s_down, int n_batches, int T, int d, int f, int E, int top_k,
                                          void* const* out_hosts, void* workspace, size_t workspace_bytes,
                                          moe_stream_t stream, moe_stream_t h2d_stream, moe_stream_t d2h_stream);
/* The same two with DeepSeek-V3's router (moe_forward_grouped_fp8 / moe_forward_grouped_fp8b as the
 * layer; bias, n_group, topk_group, scale as for moe_route_grouped). */
MOE_API int moe_forward_grouped_fp8_host_batches(const void* const* x_hosts, const float* const* logits_hosts,
                                                 const float* bias, const void* w8_gate_up, const float* s_gate_up,
                                                 const void* w8_down, const float* s_down, int n_batches, int T,
                                                 int d, int f, int E, int top_k, int n_group, int topk_group,
                                                 float scale, void* const* out_hosts, void* workspace,
                                                 size_t workspace_bytes, moe_stream_t stream, moe_stream_t h2d_stream,
                                                 moe_stream_t d2h_stream);
MOE_API int moe_forward_grouped_fp8b_host_batches(const void* const* x_hosts, const float* const* logits_hosts,
                                                  const float* bias, const void* w8_gate_up, const float* s_gate_up,
                                                  const void* w8_down, const float* s_down, int n_batches, int T,
                                                  int d, int f, int E, int top_k, int n_group, int topk_group,
                                                  float scale, void* const* out_hosts, void* workspace,
                                                  size_t workspace_bytes, moe_stream_t stream,
                                                  moe_stream_t h2d_stream, moe_stream_t d2h_stream);

/* The FP8 layers with DeepSeek-V3's router (moe_route_grouped) as step 1: bias [E] fp32, n_group,
 * topk_group and scale as for moe_route_grouped; everything else as for moe_forward_fp8 /
 * moe_forward_fp8b, with the same workspaces.  6 launches (per-row / per-channel scales; 5 with
 * MOE_FOLD_COMBINE=1) or 6–7 (blockwise, whose GEMM has no fold): routing and the permutation
 * never fuse with this router. */
MOE_API int moe_forward_grouped_fp8(const void* x, const float* logits, const float* bias, const void* w8_gate_up,
                                    const float* s_gate_up, const void* w8_down, const float* s_down, int T, int d,
                                    int f, int E, int top_k, int n_group, int topk_group, float scale, void* out,
                                    void* workspace, size_t workspace_bytes, moe_stream_t stream);
MOE_API int moe_forward_grouped_fp8b(const void* x, const float* logits, const float* bias, const void* w8_gate_up,
                                     const float* s_gate_up, const void* w8_down, const float* s_down, int T, int d,
                                     int f, int E, int top_k, int n_group, int topk_group, float scale, void* out,
                                     void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Reads (synchronously: cudaMemcpy) a device status word — a stage call's `status` pointer, or
 * the workspace of moe_forward — into *code (0 = no device-side error).  With
 * status_or_workspace = NULL it reads the status word of moe_forward_noalloc's fixed array on the
 * current device (the last noalloc call's). */
MOE_API int moe_get_device_error(const void* status_or_workspace, int32_t* code);

/* Number of kernel launches one moe_forward call makes for this shape: 4 when routing and the
 * permutation run as one kernel (E <= 32 and T*E <= 8192: each block routes every token itself to
 * build its histogram, so no grid-wide synchronisation is needed), else 5 (route, permute, two
 * grouped GEMMs, combine); 0 for T = 0; -1 for an invalid shape.  moe_forward_grouped always
 * makes 5.  In the environment, MOE_FUSE_ROUTE_PERMUTE=0 turns the route+permute fusion off (one
 * launch more) and MOE_FOLD_COMBINE=1 folds the combine into the down GEMM (one launch fewer). */
MOE_API int moe_forward_launch_count(int T, int E, int top_k);

/* Message for the last non-OK return on the calling thread ("" if none). */
MOE_API const char* moe_last_error_string(void);

/* Library version, major * 10000 + minor * 100 + patch. */
MOE_API int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
