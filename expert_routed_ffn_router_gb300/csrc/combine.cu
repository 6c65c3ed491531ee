// combine.cu -- the single-GPU counterpart of the AllToAll Combine: the weighted sum of a
// token's routed expert outputs plus the shared expert's output.
//
// Method: "Lower latency and higher throughput with multi-node DeepSeek deployment",
// section "Expert Parallelism": the results of a token's 8 routed experts are summed with
// their routing weights, and the shared expert's result is added.
//
//   Y[t, :] = sum_{j<K} topk_w[t, j] * Yp[slot_pos[t, j], :]  (+ Ysh[t, :])
//
// One CTA of 128 threads covers 1024 columns of one token; each thread owns 8 consecutive
// columns (a 16-byte bf16 vector of every routed row, two float4 of Ysh and Y).  The order
// of the additions is fixed (j ascending, then Ysh), so Y is bitwise reproducible.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int CT = 128;          // threads per CTA
constexpr int COLS = CT * 8;     // columns per CTA

__global__ void __launch_bounds__(CT) combine_kernel(const uint4 *__restrict__ Yp,
                                                     const int32_t *__restrict__ slot_pos,
                                                     const float *__restrict__ topk_w,
                                                     const float4 *__restrict__ Ysh, int H,
                                                     int K, float4 *__restrict__ Y)
{
    pdl_wait();
    // the token's K (<= 32) row numbers and weights, staged once, so that every row load of
    // a thread is issued together (one round trip instead of two per row)
    __shared__ int r_s[32];
    __shared__ float w_s[32];
    const int t = blockIdx.x;
    if (threadIdx.x < K) {
        r_s[threadIdx.x] = __ldg(slot_pos + static_cast<size_t>(t) * K + threadIdx.x);
        w_s[threadIdx.x] = __ldg(topk_w + static_cast<size_t>(t) * K + threadIdx.x);
    }
    __syncthreads();
    const int c = blockIdx.y * COLS + threadIdx.x * 8;
    if (c >= H) return;
    const unsigned n_rows = gridDim.x * static_cast<unsigned>(K);   // rows of Yp: T*K
    const int vec = H / 8;
    const int cv = c / 8;
    const size_t o = (static_cast<size_t>(t) * H + c) / 4;
    float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
    if (Ysh) {
        s0 = __ldg(Ysh + o);
        s1 = __ldg(Ysh + o + 1);
    }
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j0 = 0; j0 < K; j0 += 8) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (j0 + u < K)   // a row outside [0, T*K) (-1: a pair the dispatch rejected)
                              // contributes nothing
                v[u] = static_cast<unsigned>(r_s[j0 + u]) < n_rows
                           ? __ldg(Yp + static_cast<size_t>(r_s[j0 + u]) * vec + cv)
                           : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (j0 + u >= K) break;
            const float w = w_s[j0 + u];
            acc[0] = fmaf(w, bf16_lo(v[u].x), acc[0]);
            acc[1] = fmaf(w, bf16_hi(v[u].x), acc[1]);
            acc[2] = fmaf(w, bf16_lo(v[u].y), acc[2]);
            acc[3] = fmaf(w, bf16_hi(v[u].y), acc[3]);
            acc[4] = fmaf(w, bf16_lo(v[u].z), acc[4]);
            acc[5] = fmaf(w, bf16_hi(v[u].z), acc[5]);
            acc[6] = fmaf(w, bf16_lo(v[u].w), acc[6]);
            acc[7] = fmaf(w, bf16_hi(v[u].w), acc[7]);
        }
    }
    if (Ysh) {
        acc[0] += s0.x; acc[1] += s0.y; acc[2] += s0.z; acc[3] += s0.w;
        acc[4] += s1.x; acc[5] += s1.y; acc[6] += s1.z; acc[7] += s1.w;
    }
    Y[o] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    Y[o + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

}  // namespace

cudaError_t launch_combine(const void *Yp, const int32_t *slot_pos, const float *topk_w,
                           const float *Ysh, int T, int H, int K, float *Y, cudaStream_t s)
{
    dim3 grid(T, (H + COLS - 1) / COLS);
    return launch_pdl(combine_kernel, grid, dim3(CT), 0, s, 1, static_cast<const uint4 *>(Yp), slot_pos,
                      topk_w, reinterpret_cast<const float4 *>(Ysh), H, K, reinterpret_cast<float4 *>(Y));
}

}  // namespace moe
