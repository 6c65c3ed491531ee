// kernels.h -- host-side launchers of the library's kernels and the workspace plan.
// Internal to the library: the public boundary is include/moe.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

// ------------------------------------------------------------------------- device info
int num_sms();                 // SMs of the current device (cached per device)

// --------------------------------------------------------------------------- router
struct RouterPlan {
    int TT, TE, nTT, nET, KS, S;  // token tile, expert tile, tiles, split-K, 32-wide stages
    int max_pairs;                // shared-memory refine list capacity
    int depth;                    // summation depth of one logit (error bound)
    int gemv;                     // tiny batches: token batch (1,2,4,8) of the one-warp-per-
                                  // expert path; 0 = tile GEMM
    int split;                    // small tile GEMM, then the one-warp-per-token finalise
                                  // launch (instead of the last CTA of a token tile)
    size_t part_bytes, xsq_bytes, wsq_bytes, cnt_bytes, smem_bytes;
    size_t total() const { return part_bytes + xsq_bytes + wsq_bytes + cnt_bytes; }
};
RouterPlan router_plan(int T, int H, int E);

struct RouterScratch {
    float *part, *xsq, *wsq;
    unsigned *cnt;
};
// Routing options of other MoE families (moe_routing_t of the public header, validated).
struct RoutingOpts {
    int scoring = 0;      // 0 sigmoid, 1 softmax
    int n_group = 1;      // <= 32, divides E
    int topk_group = 1;
    int group_top = 1;    // 1 or 2
    int renorm = 1;
    bool is_default() const { return scoring == 0 && n_group == 1 && renorm == 1; }
};
cudaError_t launch_router(const void *X, const void *Wg, const float *bias, int T, int H,
                          int E, int K, int32_t *topk_idx, float *topk_w,
                          const RouterPlan &plan, const RouterScratch &scr, int *status,
                          cudaStream_t s, const RoutingOpts *ro = nullptr);

// ------------------------------------------------------------------------- dispatch
struct DispatchPlan {
    int n_chunks, n_words;             // 256-token chunks, 32-token mask rows
    size_t smask_bytes, ccnt_bytes, cbase_bytes;
    size_t total() const { return smask_bytes + ccnt_bytes + cbase_bytes; }
};
DispatchPlan dispatch_plan(int T, int E);

struct DispatchScratch {
    uint32_t *smask;
    int32_t *chunk_cnt, *chunk_base;
};
cudaError_t launch_dispatch(const void *X, const int32_t *topk_idx, int T, int H, int E,
                            int K, int32_t *counts, int32_t *offsets, int32_t *perm,
                            int32_t *slot_pos, void *Xp, int32_t *affinity,
                            const DispatchPlan &plan, const DispatchScratch &scr,
                            unsigned *zero_buf, size_t zero_n, int *status, cudaStream_t s);

// ------------------------------------------------------------------------------ fp8
// Static E4M3 quantisation of W [G][R][C] bf16 (R, C multiples of 128; R the reduction
// dimension) into Wq [G][C][R] bytes (transposed: K-major rows for the FP8 MMA) and the
// scale exponents S [G][R/128][C/128] (scale 2^S).
cudaError_t launch_quant_weight(const void *W, int G, int R, int C, void *Wq, int32_t *S,
                                cudaStream_t s);
// Quantise-dequantise bf16 rows [rows][n] (n a multiple of 128) in vectors of 128 into out
// (may alias in).
cudaError_t launch_quant_rows(const void *in, long long rows, int n, void *out, cudaStream_t s);
// bf16 rows [rows][n] in vectors of 128 -> E4M3 bytes out [rows][n] and the scales 2^k as
// fp32 sT [n / 128][rows].
cudaError_t launch_quant_rows_e4m3(const void *in, long long rows, int n, void *out, float *sT,
                                   long long ld_sT, cudaStream_t s);

// -------------------------------------------------------------------------- combine
cudaError_t launch_combine(const void *Yp, const int32_t *slot_pos, const float *topk_w,
                           const float *Ysh, int T, int H, int K, float *Y, cudaStream_t s);

// ------------------------------------------------------------------------------ FFN
// One grouped problem of the expert FFN: rows of group g are [offsets[g], offsets[g+1])
// (or one dense group of `dense_rows` rows when offsets == nullptr).
struct FfnProblem {
    const void *act;        // bf16 [rows, H] (up) -- the B operand rows
    const int32_t *offsets; // device [n_groups + 1] or nullptr
    int n_groups;
    int rows;               // extent of `act` / the outputs (tensor-map size)
    int dense_rows;         // used when offsets == nullptr
    const void *W1, *W3, *W2;  // bf16 [n_groups, H, I], [n_groups, H, I], [n_groups, I, H]
    void *h;                // bf16 [rows, I] activation scratch
    void *out;              // [rows, H] bf16 or fp32
    int out_fp32;
    // FP8: W1, W3 hold E4M3 bytes [n_groups, I, H] and W2 [n_groups, H, I] (K-major rows),
    // S1, S3 [n_groups][H/128][I/128], S2 [n_groups][I/128][H/128] the scale exponents of
    // their 128 x 128 tiles (H, I multiples of 128); `act` holds E4M3 rows [rows, H] with
    // their scales 2^k in act_s [H/128][fp8_scale_pitch(rows)] (fp32); the up projection
    // writes h (bf16) and the down projection reads its E4M3 quantisation h8 [rows, I] with
    // scales h_s [I/128][fp8_scale_pitch(rows)].  Every problem of a launch uses the same
    // format.
    int fp8;
    const int32_t *S1, *S3, *S2;
    const float *act_s;
    const void *h8;
    const float *h_s;
};

// Row pitch (in scales) of an FP8 scale table [blocks][rows]: a multiple of 4 rows, so that
// the table's row stride is a multiple of 16 bytes (a TMA requirement).
inline long long fp8_scale_pitch(long long rows) { return (rows + 3) & ~3ll; }

// Launch with programmatic stream serialization (the kernel overlaps its prologue with
// the previous kernel's tail and calls pdl_wait() before reading its inputs) and, with
// cluster_x > 1, clusters of cluster_x CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, int cluster_x, Args... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(n);
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// 0 automatic, 1 single-CTA kernel, 2 CTA-pair kernel (testing hook)
void set_ffn_variant(int v);

// Enqueues the up projection (+SwiGLU) and the down projection of up to two problems
// (the routed experts and the shared expert) that share H; I may differ per problem.  One
// persistent launch claims the up-projection tiles, then the down-projection tiles, from
// a global counter; a down tile starts once the h rows of its token tile are complete,
// tracked by `ready` (device, ffn_ready_slots(...) counters incl. the tile counter,
// zeroed here unless `ready_zeroed`).  `mid_event` (nullable) is recorded after the
// launch.
// phase_only: -1 both projections; 0 the up projections alone; 1 the down projections alone
// (after a phase-0 launch of the same problems and the same readiness counters).
// max_ctas > 0 caps the persistent grid (the rest of the GPU stays free for kernels of
// other streams); 0 takes one CTA (or CTA pair) per SM.
cudaError_t launch_ffn(const FfnProblem *probs, int n_probs, int H, const int *I_per_prob,
                       int token_hint, unsigned *ready, bool ready_zeroed, int *status, cudaStream_t s,
                       unsigned long long timeout_ns, int inject, cudaEvent_t mid_event,
                       int phase_only = -1, int max_ctas = 0);

// Readiness counters launch_ffn needs (unsigned each) for `rows` rows in `n_groups` groups
// over all its problems.
size_t ffn_ready_slots(long long rows, int n_groups);

// Raises the dynamic shared-memory limit of `func` to `bytes` once per process and size
// (a no-op afterwards, so launches stay capturable).
cudaError_t ensure_smem(const void *func, size_t bytes);

}  // namespace moe
