/*
 * moe.h -- C ABI of the GB300 (sm_103a) DeepSeek-style Mixture-of-Experts layer forward.
 *
 * The layer, as the pages describe it:
 *   "Lower latency and higher throughput with multi-node DeepSeek deployment" (Perplexity),
 *     section "Expert Parallelism": 256 routed experts and 1 shared expert; every token is
 *     sent to 8 distinct routed experts whose results are combined by a weighted sum, and
 *     the shared expert's result is added.  Dispatch sends tokens to their experts before
 *     the expert GEMMs; Combine gathers the results and forms the weighted sum.
 *     section "MoE Router": a sort that keeps the indices produces the top-k; a dense
 *     dispatch/combine needs per-expert aggregated routing information, not per-token.
 *     section "Cuda Graph" / "Quantization": kernels read the routing counts on the device
 *     instead of sizing work from buffer sizes, so a call can be captured in a CUDA graph.
 *   "DeepSeek-V4.1-Flash" vLLM article, section "Kernels", Mega-Gate: the router (gate
 *     GEMM, expert scoring, bias, top-k selection) runs as one fused kernel.
 *   "GRACE-MoE" notes, "Core Idea 1. Expert Grouping": the expert affinity matrix A of
 *     co-activations that grouping starts from; "2. Expert Replication": per-expert load W.
 *
 * Readings taken where the pages are silent (scoring = logistic sigmoid; the bias only
 * selects; ties go to the lower expert index; weights are the selected unbiased scores
 * divided by their sum; SwiGLU h = silu(x W1) * (x W3), y = h W2; shared expert weight 1)
 * are stated again at each entry point below.
 *
 * Conventions for every entry point
 *   - Every array argument is a DEVICE pointer owned by the caller, 16-byte aligned.
 *     Host structs (moe_shape_t, moe_weights_t) are read during the call only.
 *   - Row-major layouts; "bf16" arrays hold IEEE bfloat16 values (2 bytes each).
 *   - `stream` is a cudaStream_t (0 = legacy default stream).  All work is enqueued on it;
 *     no call synchronises the host (moe_read_status, and every call in the debug mode of
 *     moe_debug_set_sync_status, excepted), allocates or frees memory, so calls can be
 *     captured in a CUDA graph.  Outputs are valid once the stream reaches them.  (One exception,
 *     moe_layer_forward on bf16 weights up to 128 tokens: it forks the shared expert onto a
 *     side stream of the library and joins it back before the combine; that stream and
 *     its two events are created by the first such call of a host thread on a device and
 *     released when that thread exits.)
 *   - `ws` is a caller-owned device workspace of at least moe_workspace_bytes() bytes
 *     (256-byte aligned).  Its first 4 bytes are the status word: zero them once after
 *     allocating (e.g. cudaMemset); moe_read_status() resets the word after reading it.
 *     Calls that share a workspace must be serialised by the caller.
 *   - Arguments are validated on the host before anything is enqueued: an invalid call
 *     returns a negative moe_status_t and has no effect.  A failing launch returns
 *     MOE_ERR_CUDA.  Conditions found on the device (a bounded wait that ran out, an
 *     expert index outside [0, E) given to moe_dispatch, group offsets outside [0, rows]
 *     given to moe_expert_ffn) are recorded in the workspace's status word and never lead
 *     to an access out of bounds; read them with moe_read_status().
 *   - Supported shapes: 1 <= E <= 1024, 1 <= K <= min(E, 32), H and I multiples of 64,
 *     T >= 0 (T == 0 enqueues nothing and returns MOE_OK), T*K < 2^31.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,        /* null pointer, negative size, K > E, ...; on the
                                        device: out-of-range expert index or offsets      */
    MOE_ERR_UNSUPPORTED_SHAPE = -2,  /* H or I not a multiple of 64, E > 1024, K > 32, ... */
    MOE_ERR_MISALIGNED = -3,         /* a pointer is not 16-byte aligned (ws: 256-byte)     */
    MOE_ERR_WORKSPACE_TOO_SMALL = -4,
    MOE_ERR_CUDA = -5,               /* a CUDA runtime/driver call failed                  */
    MOE_ERR_DEVICE_TIMEOUT = -6,     /* a bounded device-side wait ran out (status word)   */
    MOE_ERR_NOT_IMPLEMENTED = -7
} moe_status_t;

/* Layer shape.  T tokens, hidden size H, E routed experts, top-K, expert intermediate
 * size I, shared-expert intermediate size I_shared (0 = no shared expert). */
typedef struct moe_shape {
    int32_t T, H, E, K, I, I_shared;
} moe_shape_t;

/* Layer weights (device pointers).
 *   W_gate bf16 [E, H]      router gate rows
 *   bias   fp32 [E]         per-expert selection bias (selection only, not in the weights)
 *   W1     bf16 [E, H, I]   gate projection of each routed expert (I contiguous)
 *   W3     bf16 [E, H, I]   up projection
 *   W2     bf16 [E, I, H]   down projection (H contiguous)
 *   W1s, W3s bf16 [H, I_shared], W2s bf16 [I_shared, H]: the shared expert (NULL when
 *   I_shared == 0). */
typedef struct moe_weights {
    const void *W_gate;
    const float *bias;
    const void *W1, *W3, *W2;
    const void *W1s, *W3s, *W2s;
} moe_weights_t;

/* Layer weights with FP8 experts ("Lower latency and higher throughput...", Quantization:
 * weights quantised ahead of time with one scale per 128 x 128 tile).  W_gate and bias as in
 * moe_weights_t (the router is not quantised).  W1, W3 hold E4M3 bytes [E, I, H] and W2
 * [E, H, I] (W1s, W3s [I_shared, H], W2s [H, I_shared]): each matrix of moe_weights_t
 * TRANSPOSED, so that every output column's reduction values are contiguous (the K-major
 * rows the FP8 tensor-core MMA reads).  S1, S3 int32 [E, H/128, I/128] and S2 int32
 * [E, I/128, H/128] (S1s, S3s [H/128, I_shared/128], S2s [I_shared/128, H/128]) hold the
 * scale exponents, indexed as the untransposed matrices' 128 x 128 tiles: a weight is its
 * E4M3 value times 2^S of its tile.  moe_quantize_weight_fp8 produces both from bf16
 * weights. */
typedef struct moe_weights_fp8 {
    const void *W_gate;
    const float *bias;
    const void *W1, *W3, *W2;
    const int32_t *S1, *S3, *S2;
    const void *W1s, *W3s, *W2s;
    const int32_t *S1s, *S3s, *S2s;
} moe_weights_fp8_t;

/* Bytes of workspace that moe_layer_forward needs for `shape`; it also suffices for every
 * other entry point called with the same or smaller sizes.  Returns 0 for an invalid shape. */
size_t moe_workspace_bytes(const moe_shape_t *shape);

/* Where moe_layer_forward keeps its intermediate results inside the workspace: byte
 * offsets from `ws` of offsets int32 [E + 1], perm int32 [T*K], slot_pos int32 [T, K] (the
 * dispatch bookkeeping, as moe_dispatch defines it), Xp bf16 [T*K, H] (the permuted token
 * rows), h bf16 [T*K, I] (the SwiGLU activations), Yp bf16 [T*K, H] (the expert outputs)
 * and Ysh fp32 [T, H] (the shared expert's output; 0 when I_shared == 0), and `bytes` =
 * moe_workspace_bytes(shape).  They hold what the last layer call on that workspace left
 * there, once its stream has reached the end of the call (with FP8 experts, h and Yp hold
 * the bf16 activations and outputs the FP8 GEMMs read and wrote; their E4M3 operands live
 * elsewhere in the workspace).  For inspection and testing; not on the pages.  Returns MOE_OK, or MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED_SHAPE for a
 * shape moe_workspace_bytes rejects. */
typedef struct moe_workspace_layout {
    size_t offsets, perm, slot_pos, Xp, h, Yp, Ysh, bytes;
} moe_workspace_layout_t;
int moe_workspace_layout(const moe_shape_t *shape, moe_workspace_layout_t *out);

/* Static, NUL-terminated description of a moe_status_t value. */
const char *moe_error_string(int status);

/* Reads the device status word of workspace `ws` (synchronising `stream`), resets it to
 * MOE_OK and returns what it held: MOE_OK, MOE_ERR_DEVICE_TIMEOUT (a bounded device-side
 * wait ran out) or MOE_ERR_INVALID_ARG (the dispatch met an expert index outside [0, E),
 * or the expert FFN group offsets outside [0, rows]); MOE_ERR_CUDA if the copy itself
 * failed. */
int moe_read_status(void *ws, void *stream);

/* Debugging hook: with on = 1, every later call that records device-side conditions in a
 * workspace status word (moe_router_topk, moe_router_topk_ex, moe_dispatch,
 * moe_expert_ffn, moe_layer_forward, moe_layer_forward_ex, moe_layer_forward_fp8)
 * synchronises its stream after enqueueing its work and returns that word, read and reset
 * as by moe_read_status, in place of MOE_OK -- except for an empty batch and inside a stream
 * capture (a capture cannot be synchronised).  on = 0 (the default) restores the
 * asynchronous calls.  Process-wide; not for production use: it serialises the host with
 * the GPU. */
void moe_debug_set_sync_status(int on);

/* Testing hook: sets the limit of the bounded device-side waits of the tensor-core FFN
 * kernels (0 restores the default of one second) and, with inject_stall = 1, makes their
 * TMA producer skip its work so that the waits run out and MOE_ERR_DEVICE_TIMEOUT is
 * recorded in the status word (no fault, no hang).  Affects later moe_expert_ffn and
 * moe_layer_forward calls of the process; not for production use. */
void moe_debug_set_wait_limit(unsigned long long limit_ns, int inject_stall);

/* Profiling hook: with `events` pointing at n >= 6 cudaEvent_t handles, every later
 * moe_layer_forward records them on its stream: [0] before the router, [1] after the
 * router, [2] after dispatch, [3] and [4] after the expert FFN (its up and down
 * projections are one launch), [5] after combine.  events == NULL switches recording off.  The
 * handles stay owned by the caller and must outlive the recording calls. */
void moe_debug_set_stage_events(void *const *events, int n);

/* Testing hook: which expert-FFN kernel later moe_expert_ffn and moe_layer_forward calls
 * of the process launch.  0 (the default) chooses by token tile: tiles of 128 rows or more
 * run on CTA pairs (256-row weight tiles, 2-SM tensor-core MMA), smaller ones on single
 * CTAs (128-row weight tiles).  1 forces single CTAs, 2 forces CTA pairs.  Both give the
 * same results; other values act as 0.  Not for production use. */
void moe_debug_set_ffn_variant(int variant);

/* Testing hook: where later moe_layer_forward calls on bf16 weights run the shared expert.
 * -1 (the default) chooses by batch size: up to 128 tokens it runs as its own FFN launch on
 * a quarter of the SMs, on a side stream of the library forked from the caller's stream before
 * the router and joined back before the combine, so that it overlaps the router and the
 * dispatch; larger batches run it in the routed experts' launch.  0 always takes the
 * routed experts' launch, 1 always the side stream.  Same results either way; other
 * values act as -1.  Not for production use. */
void moe_debug_set_shared_side(int mode);

/* Router: gate GEMM, sigmoid scoring, selection bias, top-K, renormalised weights
 * ("DeepSeek-V4.1-Flash", Kernels, Mega-Gate: fused into one kernel; "Lower latency and
 * higher throughput...", MoE Router).  One launch up to 15 tokens and from 2049 to 4096
 * tokens (the last CTA of each token tile selects; up to ~800 experts, whose per-warp
 * arrays fit that CTA's shared memory); other batches take a tile-GEMM
 * launch that leaves split-K partial logits in the workspace and a finalise launch that
 * sums, scores and selects them (the scores themselves are never stored).
 *   X      bf16 [T, H]      token activations
 *   W_gate bf16 [E, H]
 *   bias   fp32 [E]
 *   out topk_idx int32 [T, K]: the K experts with the largest sel = sigmoid(X W_gate^T) +
 *       bias, in descending sel order, equal sel -> lower index first.  The selection is
 *       the one exact arithmetic gives: fp32 scores carry a rigorous error bound and any
 *       token whose order the bound cannot certify is re-scored in double-word arithmetic.
 *       A token whose row of X (or a gate row) holds a NaN, an infinity or values whose
 *       products overflow has no defined selection; it still gets K distinct experts in
 *       [0, E) (its weights may be NaN), and the call does not fail.
 *   out topk_w fp32 [T, K]: s_j / sum_j s_j over the selected unbiased scores s.
 *   ws / ws_bytes: workspace (split-K partial logits, completion counters). */
int moe_router_topk(const void *X, const void *W_gate, const float *bias,
                    int T, int H, int E, int K,
                    int32_t *topk_idx, float *topk_w,
                    void *ws, size_t ws_bytes, void *stream);

/* Routing options of the other MoE families one router serves ("Lower latency and higher
 * throughput...", MoE Router: one router for every MoE model, DeepSeek's routing selects
 * among expert groups and Mixtral's is the case of a single group holding every expert).
 * The defaults {0, 1, 1, 1, 1} are moe_router_topk's routing.  A NULL moe_routing_t
 * pointer means the defaults. */
typedef struct moe_routing {
    int scoring;     /* 0: s = sigmoid(l); 1: s = softmax of the token's E logits */
    int n_group;     /* the E experts form n_group groups of E / n_group consecutive
                        experts (n_group divides E; 1..32; 1 = no group limit) */
    int topk_group;  /* groups kept per token (1..n_group): those with the largest group
                        score, equal scores -> lower group first; the top-K is taken among
                        their experts only */
    int group_top;   /* a group's score is the sum of its group_top (1 or 2) largest
                        sel = s + bias */
    int renorm;      /* 1: topk_w = the selected s divided by their sum; 0: the selected s */
} moe_routing_t;

/* moe_router_topk with routing options.  Selection order, tie-breaks and exactness as for
 * moe_router_topk (a token the fp32 bounds cannot certify is re-scored for every expert
 * in double-word arithmetic).  Errors: MOE_ERR_INVALID_ARG when the options define no
 * selection (n_group not dividing E, topk_group outside 1..n_group, K > topk_group * E /
 * n_group, scoring or renorm not 0/1, group_top < 1 or > E / n_group);
 * MOE_ERR_UNSUPPORTED_SHAPE for n_group > 32 or group_top > 2. */
int moe_router_topk_ex(const void *X, const void *W_gate, const float *bias,
                       int T, int H, int E, int K, const moe_routing_t *routing,
                       int32_t *topk_idx, float *topk_w,
                       void *ws, size_t ws_bytes, void *stream);

/* Router for callers that cannot allocate device memory.  No counterpart on the pages:
 * this is a convenience of this library.  Same inputs, outputs and results as
 * moe_router_topk, but without a workspace argument: the scratch lives in a fixed 16 MiB
 * array that the library holds on every GPU that loads it, until the process exits.
 * Meant for code that may not call cudaMalloc or a framework allocator -- a plug-in
 * whose host application owns all device memory and hands out only the input and output
 * buffers, or a path whose allocator is frozen after start-up.
 *   - The first call on a device looks up the array's device address (with that device
 *     current) and caches it together with the id of the device's context; make that
 *     first call before any stream capture.  If the context is destroyed and created again
 *     (cudaDeviceReset), the next call sees the new context id and looks the address up
 *     again.
 *   - Allocates and frees nothing.  Shapes whose router scratch does not fit in 16 MiB
 *     return MOE_ERR_UNSUPPORTED_SHAPE before anything is enqueued (every T <= 2048 with
 *     E <= 256 and H <= 7168 fits).
 *   - All calls on a device share the one array and it keeps what the last call left;
 *     the part that must start at zero is cleared on `stream` by every call.  Calls whose
 *     work overlaps on the GPU (other streams, other host threads) race on the array:
 *     serialise them.
 *   - Conditions found on the device (a bounded wait of the large-batch router kernel that
 *     ran out: MOE_ERR_DEVICE_TIMEOUT) go to a status word inside the array, which only
 *     moe_router_topk_noalloc_status reads. */
int moe_router_topk_noalloc(const void *X, const void *W_gate, const float *bias,
                            int T, int H, int E, int K,
                            int32_t *topk_idx, float *topk_w, void *stream);

/* Status word of moe_router_topk_noalloc on the current device: synchronises `stream`,
 * returns what the word held (MOE_OK or MOE_ERR_DEVICE_TIMEOUT; MOE_ERR_CUDA if the copy
 * failed) and resets it to MOE_OK.  Like moe_read_status, but for the library's own array
 * (no workspace); allocates nothing.  Not on the pages. */
int moe_router_topk_noalloc_status(void *stream);

/* Dispatch: the single-GPU counterpart of the AllToAll Dispatch ("Lower latency and higher
 * throughput...", Expert Parallelism; MoE Router: per-expert aggregated routing info).
 *   X        bf16 [T, H], topk_idx int32 [T, K] (values in [0, E), distinct per token)
 *   out counts   int32 [E]      tokens routed to each expert (the per-expert load W of
 *                               "GRACE-MoE", Expert Replication)
 *   out offsets  int32 [E + 1]  exclusive prefix sum of counts; offsets[E] = T*K
 *   out perm     int32 [T*K]    token of permuted row r; rows are ordered by
 *                               (expert ascending, token ascending) -- deterministic
 *   out slot_pos int32 [T, K]   permuted row that holds (token t, slot j)
 *   out Xp       bf16 [T*K, H]  Xp[r] = X[perm[r]]
 *   out affinity int32 [E, E]   (nullable) tokens whose top-K holds both i and j, zero
 *                               diagonal ("GRACE-MoE", Expert Grouping, matrix A)
 *   ws / ws_bytes: workspace (per-token-group expert bit masks and counts).
 * An index outside [0, E) is recorded as MOE_ERR_INVALID_ARG in the workspace's status word
 * (moe_read_status); its pair gets no row (slot_pos = -1, left out of counts, perm, Xp and
 * affinity, so offsets[E] < T*K) and nothing is written out of bounds. */
int moe_dispatch(const void *X, const int32_t *topk_idx, int T, int H, int E, int K,
                 int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *slot_pos,
                 void *Xp, int32_t *affinity,
                 void *ws, size_t ws_bytes, void *stream);

/* Grouped SwiGLU expert FFN over expert-contiguous rows ("Lower latency and higher
 * throughput...", Roofline / GroupGEMM: group i has m_i rows, [m_i, k] x [k, n];
 * Quantization: SiLU-and-multiply activation).  For group g, rows r in
 * [offsets[g], offsets[g+1]):
 *     Yp[r] = ( silu(Xp[r] W1[g]) * (Xp[r] W3[g]) ) W2[g]
 * tcgen05 tensor cores with fp32 accumulation; the activation h is rounded to bf16.
 *   Xp      bf16 [rows, H]
 *   offsets int32 [n_groups + 1] on the device, non-decreasing, offsets[0] = 0,
 *           offsets[n_groups] <= rows; read by the kernels, never by the host (offsets
 *           that decrease or leave [0, rows] are recorded as MOE_ERR_INVALID_ARG in the
 *           status word and no tile runs: nothing is written)
 *   W1, W3  bf16 [n_groups, H, I];  W2 bf16 [n_groups, I, H]
 *   out Yp  [rows, H], bf16 (out_fp32 == 0) or fp32 (out_fp32 == 1)
 *   rows    upper bound of offsets[n_groups] (sizes the tensor maps and the workspace)
 *   ws / ws_bytes: at least moe_expert_ffn_workspace_bytes(rows, n_groups, I) bytes (the
 *           bf16 activation h [rows, I] and per-token-tile completion counters).
 * The shared expert is the case n_groups = 1, offsets = {0, T}. */
/* Workspace bytes moe_expert_ffn needs for `rows` rows in `n_groups` groups of
 * intermediate size I (0 for invalid arguments).  Not on the pages: a sizing helper. */
size_t moe_expert_ffn_workspace_bytes(int rows, int n_groups, int I);

int moe_expert_ffn(const void *Xp, const int32_t *offsets, int n_groups, int rows,
                   int H, int I,
                   const void *W1, const void *W3, const void *W2,
                   void *Yp, int out_fp32,
                   void *ws, size_t ws_bytes, void *stream);

/* Combine: the single-GPU counterpart of the AllToAll Combine ("Lower latency and higher
 * throughput...", Expert Parallelism: weighted sum of the routed results plus the shared
 * expert's result).
 *     Y[t] = sum_j topk_w[t, j] * Yp[slot_pos[t, j]]  (+ Ysh[t] when Ysh != NULL)
 *   Yp bf16 [T*K, H], slot_pos int32 [T, K], topk_w fp32 [T, K], Ysh fp32 [T, H] or NULL
 *   out Y fp32 [T, H].  Summation order is fixed (j ascending, then Ysh).  A slot_pos entry
 * outside [0, T*K) -- -1 marks a pair moe_dispatch rejected -- contributes nothing. */
int moe_combine(const void *Yp, const int32_t *slot_pos, const float *topk_w,
                const float *Ysh, int T, int H, int K, float *Y, void *stream);

/* Whole layer: router -> dispatch -> grouped expert FFN and shared expert -> combine.
 * Up to 128 tokens on bf16 weights the shared expert runs on the library's side stream
 * beside the router and the dispatch (joined back into `stream` before the combine).
 *   X bf16 [T, H]; out Y fp32 [T, H]
 *   out topk_idx int32 [T, K], topk_w fp32 [T, K], counts int32 [E] (required)
 *   out affinity int32 [E, E] (nullable: skipped when NULL)
 *   ws / ws_bytes: at least moe_workspace_bytes(shape). */
int moe_layer_forward(const moe_shape_t *shape, const moe_weights_t *weights,
                      const void *X, float *Y,
                      int32_t *topk_idx, float *topk_w, int32_t *counts,
                      int32_t *affinity,
                      void *ws, size_t ws_bytes, void *stream);

/* moe_layer_forward with routing options (moe_routing_t; NULL = the defaults, the same
 * call as moe_layer_forward).  Same workspace; option errors as moe_router_topk_ex. */
int moe_layer_forward_ex(const moe_shape_t *shape, const moe_weights_t *weights,
                         const moe_routing_t *routing, const void *X, float *Y,
                         int32_t *topk_idx, float *topk_w, int32_t *counts,
                         int32_t *affinity,
                         void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------------------
 * FP8 experts ("Lower latency and higher throughput...", Quantization: FP8 with block-wise
 * scales, weights per 128 x 128 tile ahead of time, activations per 128-element vector on
 * the fly).  Format E4M3 (largest finite 448), round to nearest even; a block's scale is
 * the power of two 2^k with k the smallest integer such that amax <= 448 * 2^k (0 for an
 * all-zero block), clamped to [-124, 127], so every dequantised value q * 2^k is exact in
 * bf16.
 * ------------------------------------------------------------------------------------ */

/* Static weight quantisation: W bf16 [G, R, C] (R, C multiples of 128, else
 * MOE_ERR_UNSUPPORTED_SHAPE; R is the reduction dimension: H for W1 / W3, I for W2) -> Wq
 * E4M3 bytes [G, C, R] (transposed) and S int32 [G, R/128, C/128] (the tile's k).  Device
 * pointers, enqueued on `stream`. */
int moe_quantize_weight_fp8(const void *W, int G, int R, int C, void *Wq, int32_t *S,
                            void *stream);

/* Activation quantisation as the FP8 layer applies it: every row of `in` bf16 [rows, n]
 * (n a multiple of 128) in vectors of 128, quantised to E4M3 and dequantised back, into
 * `out` bf16 [rows, n] (out may equal in).  Device pointers, enqueued on `stream`. */
int moe_quantize_rows_fp8(const void *in, long long rows, int n, void *out, void *stream);

/* The layer with FP8 experts: as moe_layer_forward_ex, with the expert FFNs (routed and
 * shared) computed from the E4M3 weights and their tile scales on token rows quantised in
 * vectors of 128 along H and on h = silu(x W1) * (x W3), rounded to bf16, quantised in
 * vectors of 128 along I.  The tensor cores multiply the E4M3 values (FP8 MMA) one
 * 128-wide block of the reduction at a time; each block's fp32 partial sum is scaled by
 * the block's weight and activation scales (powers of two) and added in fp32.  H, I and
 * I_shared must be multiples of 128 and at most 16384 (else MOE_ERR_UNSUPPORTED_SHAPE).
 * Same workspace as moe_layer_forward. */
int moe_layer_forward_fp8(const moe_shape_t *shape, const moe_weights_fp8_t *weights,
                          const moe_routing_t *routing, const void *X, float *Y,
                          int32_t *topk_idx, float *topk_w, int32_t *counts,
                          int32_t *affinity,
                          void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------------------
 * GRACE-MoE placement planner ("GRACE-MoE" notes, Core Idea 1-3).  Host code on HOST
 * pointers: it consumes the counts and the affinity matrix moe_layer_forward produces
 * (copied to the host by the caller) and plans where experts go for expert parallelism
 * over D GPUs.  Plain C arrays in, plain C arrays out; the planner allocates host memory
 * for its own scratch only, never device memory.  All calls validate their arguments and
 * return MOE_ERR_INVALID_ARG without writing anything when they do not hold.
 * ------------------------------------------------------------------------------------ */

/* Core Idea 1: U = affinity inside groups / all affinity, over the pairs i < j of the
 * symmetric affinity [E, E]; S = sqrt(mean over the D groups of (|C_d| - E/D)^2).
 * group_of [E] holds group ids 0..D-1. */
int moe_grace_metrics(const int32_t *affinity, int E, const int32_t *group_of, int D,
                      double *U, double *S);

/* Core Idea 1: spectral grouping of the E experts into D groups whose sizes stay within
 * [ceil(E/D - delta), floor(E/D + delta)], delta = (E/D) r (r >= 0; the bounds must admit
 * a partition).  Normalised spectral embedding (the D leading eigenvectors of
 * Deg^-1/2 A Deg^-1/2, rows scaled to unit length) and a size-bounded k-means from
 * farthest-point seeds.  out group_of [E].  E <= 4096 (cost O(E^3)). */
int moe_grace_group(const int32_t *affinity, int E, int D, double r, int32_t *group_of);

/* Core Idea 1: moe_grace_group at every r of the increasing grid r_grid [n_r]; out U, S
 * [n_r] (the metrics of each grouping), *knee (the grid index where U and r scaled to
 * [0, 1] differ most: beyond it a looser size bound buys less affinity than on average)
 * and group_of [E] (the grouping at the knee). */
int moe_grace_choose_r(const int32_t *affinity, int E, int D, const double *r_grid, int n_r,
                       double *U, double *S, int *knee, int32_t *group_of);

/* Core Idea 2: replication of the heaviest group's hot experts. */
typedef struct moe_grace_replication {
    int heaviest;        /* group (GPU) with the largest load W_max; ties -> lower id */
    int n_replica;       /* min(max(1, floor(rho)), D - 1) */
    int n_hot;           /* hot experts written to hot[0 .. n_hot) */
    double rho;          /* W_max / W_mean */
    double W_mean;
    long long W_max;
    long long W_r;       /* load of the hot experts */
} moe_grace_replication_t;

/* counts [E] (expert loads, e.g. moe_layer_forward's counts), group_of [E] (D >= 2 groups);
 * out W [D] (group loads), hot [E] (the heaviest group's experts by load, descending, ties
 * -> lower index, until their cumulative load exceeds W_max * n_replica / (1 + n_replica)),
 * replica_gpus [D - 1] (the first n_replica written: the least-loaded other GPUs, ties ->
 * lower id), *out. */
int moe_grace_replicate(const int32_t *counts, int E, const int32_t *group_of, int D,
                        long long *W, int32_t *hot, int32_t *replica_gpus,
                        moe_grace_replication_t *out);

/* Core Idea 3: instance weights of a hot expert.  Instances: [rep->heaviest] followed by
 * replica_gpus[0 .. n_replica).  out predicted [1 + n_replica]: W_max - W_r + W_p for the
 * original, W_i + W_p for a copy on GPU i, W_p = W_r / (1 + n_replica).  out table
 * [D][1 + n_replica]: for a token on GPU src, the probability of each instance -- weights
 * proportional to 1 / predicted, over the instances on src if any, else those on src's
 * node (gpus_per_node consecutive GPU ids per node), else all instances. */
int moe_grace_route_table(const long long *W, int D, const moe_grace_replication_t *rep,
                          const int32_t *replica_gpus, int gpus_per_node, double *predicted,
                          double *table);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
