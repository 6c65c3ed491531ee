// router.cu -- fused MoE router: gate GEMM -> sigmoid scoring -> selection bias -> top-k
// -> renormalised weights, in one kernel.
//
// Method: "DeepSeek-V4.1-Flash" (vLLM article), section "Kernels", Mega-Gate: the gate
// GEMM, expert scoring, bias and top-k selection run in one kernel instead of a GEMM plus
// a separate top-k kernel with a round trip of the scores.  "Lower latency and higher
// throughput with multi-node DeepSeek deployment", section "MoE Router": the top-k is a
// sort that keeps the expert indices.
//
// Scoring reading: s = sigmoid(l), l = x . W_gate[e]; the selection key is sel = s + b[e];
// order is sel descending with equal sel going to the lower expert index; the weights are
// the selected s divided by their sum (the bias does not enter the weights).
//
// Exactness.  The selection must be the one exact arithmetic gives.  bf16 x bf16 products
// are exact in fp32, so the only error of the fp32 logit is the rounding of its sums.  The
// summation here is a fixed tree in which every product passes through at most d
// additions, so |l_fp32 - l| <= gamma_d * sum|x_h w_h| <= gamma_d * ||x|| * ||w||
// (Cauchy-Schwarz), gamma_d = d u / (1 - d u), u = 2^-24.  Propagating that bound through
// the sigmoid and the bias add gives an interval per expert.  When the intervals certify
// both the chosen set and its order, the fp32 result is exact; otherwise every expert
// whose interval reaches the k-th lower bound is re-scored in double-word fp32 arithmetic
// (error-free TwoSum accumulation of the exact products, ~2^-48 relative) with an fp64
// sigmoid, and the top-k is taken again among those candidates.
//
// Structure.  Grid (expert tiles, token tiles, K splits).  Each CTA computes a 64x64
// tile of fp32 logits over its slice of H on the CUDA cores and writes it to the
// workspace; the last CTA of a token tile (completion counter) sums the split-K partials in
// a fixed order, scores, selects and writes the outputs -- one launch, no host sync.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int TT = 64;     // tokens per CTA tile
constexpr int TE = 64;     // experts per CTA tile
constexpr int KST = 32;    // k per shared-memory stage
constexpr int NT = 256;    // threads
constexpr int NW = NT / 32;
constexpr float kU = 5.9604644775390625e-8f;  // 2^-24

struct RouterArgs {
    const uint16_t *X, *Wg;
    const float *bias;
    int T, H, E, K, KS, S;
    float *part;     // [KS][T][E]
    float *xsq;      // [KS][T]
    float *wsq;      // [nTT][KS][E]
    unsigned *cnt;   // [nTT]
    int32_t *topk_idx;
    float *topk_w;
    int *status;
};

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// (sel, e) ranks before (sel2, e2): larger sel, then lower index.
__device__ __forceinline__ bool before(float a, int ea, float b, int eb)
{
    return a > b || (a == b && ea < eb);
}
__device__ __forceinline__ bool before64(double a, int ea, double b, int eb)
{
    return a > b || (a == b && ea < eb);
}

// Error-free transformation: s + err == a + b exactly (Knuth's TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &err)
{
    s = __fadd_rn(a, b);
    float bp = __fsub_rn(s, a);
    float ap = __fsub_rn(s, bp);
    err = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

// Double-word dot product of a bf16 token row and a bf16 gate row, reduced over the warp
// in a fixed order; every lane returns the same value.
__device__ double dot_double_word(const uint16_t *x, const uint16_t *w, int H, int lane)
{
    const uint4 *xr = reinterpret_cast<const uint4 *>(x);
    const uint4 *wr = reinterpret_cast<const uint4 *>(w);
    float hi = 0.f, lo = 0.f;
    for (int v = lane; v < H / 8; v += 32) {
        float xf[8], wf[8];
        unpack8(xr[v], xf);
        unpack8(wr[v], wf);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float p = __fmul_rn(xf[i], wf[i]);  // exact: 8-bit x 8-bit significands
            float s, e;
            two_sum(hi, p, s, e);
            hi = s;
            lo = __fadd_rn(lo, e);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float ohi = __shfl_xor_sync(kFullMask, hi, off);
        float olo = __shfl_xor_sync(kFullMask, lo, off);
        float s, e;
        two_sum(hi, ohi, s, e);
        hi = s;
        lo = __fadd_rn(__fadd_rn(lo, olo), e);
    }
    return static_cast<double>(hi) + static_cast<double>(lo);
}

__global__ void __launch_bounds__(NT, 2) router_kernel(const RouterArgs a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_last;

    const int et = blockIdx.x, tt = blockIdx.y, ks = blockIdx.z;
    const int nET = gridDim.x;
    const int tid = threadIdx.x;
    const int t0 = tt * TT, e0 = et * TE;
    const int s_beg = static_cast<int>(static_cast<long long>(ks) * a.S / a.KS);
    const int s_end = static_cast<int>(static_cast<long long>(ks + 1) * a.S / a.KS);

    // ------------------------------------------------------------------ tile GEMM
    float *xs = reinterpret_cast<float *>(smem);   // [2][KST][TT]
    float *wsm = xs + 2 * KST * TT;                // [2][KST][TE]

    const int lr = tid & 63, lv = tid >> 6;        // loader: row, 8-element vector
    const int xrow = t0 + lr, wrow = e0 + lr;
    const bool xok = xrow < a.T, wok = wrow < a.E;
    const uint4 *xp = reinterpret_cast<const uint4 *>(a.X + static_cast<size_t>(xok ? xrow : 0) * a.H) + lv;
    const uint4 *wp = reinterpret_cast<const uint4 *>(a.Wg + static_cast<size_t>(wok ? wrow : 0) * a.H) + lv;
    float xsq = 0.f, wsq = 0.f;
    uint4 xr = make_uint4(0, 0, 0, 0), wr = make_uint4(0, 0, 0, 0);

    const int tx = tid & 15, ty = tid >> 4;        // compute: experts 4tx.., tokens 4ty..
    float acc_mid[16], acc_out[16];
#pragma unroll
    for (int p = 0; p < 16; ++p) { acc_mid[p] = 0.f; acc_out[p] = 0.f; }

    auto gload = [&](int s) {
        xr = xok ? __ldg(xp + s * 4) : make_uint4(0, 0, 0, 0);
        wr = wok ? __ldg(wp + s * 4) : make_uint4(0, 0, 0, 0);
    };
    auto sstore = [&](int buf) {
        float xf[8], wf[8];
        unpack8(xr, xf);
        unpack8(wr, wf);
        float *xd = xs + buf * KST * TT + (lv * 8) * TT + lr;
        float *wd = wsm + buf * KST * TE + (lv * 8) * TE + lr;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            xd[i * TT] = xf[i];
            wd[i * TE] = wf[i];
            xsq = fmaf(xf[i], xf[i], xsq);
            wsq = fmaf(wf[i], wf[i], wsq);
        }
    };

    if (s_beg < s_end) {
        gload(s_beg);
        sstore(0);
    }
    __syncthreads();
    int buf = 0, nmid = 0;
    for (int s = s_beg; s < s_end; ++s) {
        if (s + 1 < s_end) gload(s + 1);
        float acc_in[16];
#pragma unroll
        for (int p = 0; p < 16; ++p) acc_in[p] = 0.f;
        const float *xb = xs + buf * KST * TT + 4 * ty;
        const float *wb = wsm + buf * KST * TE + 4 * tx;
#pragma unroll 8
        for (int kk = 0; kk < KST; ++kk) {
            const float4 xv = *reinterpret_cast<const float4 *>(xb + kk * TT);
            const float4 wv = *reinterpret_cast<const float4 *>(wb + kk * TE);
            const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
            const float wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc_in[i * 4 + j] = fmaf(xa[i], wa[j], acc_in[i * 4 + j]);
        }
#pragma unroll
        for (int p = 0; p < 16; ++p) acc_mid[p] += acc_in[p];
        if (++nmid == 8) {
#pragma unroll
            for (int p = 0; p < 16; ++p) { acc_out[p] += acc_mid[p]; acc_mid[p] = 0.f; }
            nmid = 0;
        }
        if (s + 1 < s_end) sstore(buf ^ 1);
        __syncthreads();
        buf ^= 1;
    }
#pragma unroll
    for (int p = 0; p < 16; ++p) acc_out[p] += acc_mid[p];

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + 4 * ty + i;
        if (t >= a.T) continue;
        float *dst = a.part + (static_cast<size_t>(ks) * a.T + t) * a.E;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + 4 * tx + j;
            if (e < a.E) dst[e] = acc_out[i * 4 + j];
        }
    }

    // squared norms of this slice, reduced over the 4 loader threads of a row in order
    {
        float *rx = xs;            // [4][64]
        float *rw = xs + 4 * 64;   // [4][64]
        rx[lv * 64 + lr] = xsq;
        rw[lv * 64 + lr] = wsq;
        __syncthreads();
        if (tid < 64) {
            const float sx = ((rx[tid] + rx[64 + tid]) + rx[128 + tid]) + rx[192 + tid];
            const float sw = ((rw[tid] + rw[64 + tid]) + rw[128 + tid]) + rw[192 + tid];
            if (et == 0 && t0 + tid < a.T) a.xsq[static_cast<size_t>(ks) * a.T + t0 + tid] = sx;
            if (e0 + tid < a.E)
                a.wsq[(static_cast<size_t>(tt) * a.KS + ks) * a.E + e0 + tid] = sw;
        }
    }

    // ------------------------------------------------------------ last CTA finalises
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&a.cnt[tt], 1u);
        s_last = (prev == static_cast<unsigned>(nET * a.KS - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    const int warp = tid >> 5, lane = tid & 31;
    const int E = a.E, K = a.K, KS = a.KS;
    const int NI = (E + 31) / 32;
    // per-warp arrays: sel[E], bnd[E], sc[E] (fp32) and sel64[E] (fp64)
    float *w_sel = reinterpret_cast<float *>(smem) + static_cast<size_t>(warp) * 3 * E;
    float *w_bnd = w_sel + E;
    float *w_sc = w_bnd + E;
    double *w_s64 = reinterpret_cast<double *>(
        smem + static_cast<size_t>(NW) * 3 * E * sizeof(float)) + static_cast<size_t>(warp) * E;
    int *w_ord = reinterpret_cast<int *>(
        smem + static_cast<size_t>(NW) * 3 * E * sizeof(float) +
        static_cast<size_t>(NW) * E * sizeof(double)) + warp * 32;

    // depth of the summation tree (see the file comment) and the norm inflation
    const int ns_max = (a.S + KS - 1) / KS;
    const float depth = static_cast<float>(KST + 8 + (ns_max + 7) / 8 + 1 + KS + 2);
    const float gam = depth * kU / (1.f - depth * kU) * 1.0001f;
    const float infl = 1.f + static_cast<float>(a.H + 16 + KS) * (2.f * kU) + 4.f * kU;

    for (int tl = warp; tl < TT; tl += NW) {
        const int t = t0 + tl;
        if (t >= a.T) break;
        float nx2 = 0.f;
        for (int q = 0; q < KS; ++q) nx2 += a.xsq[static_cast<size_t>(q) * a.T + t];
        const float nx = sqrtf(nx2) * infl;

        for (int i = 0; i < NI; ++i) {
            const int e = lane + 32 * i;
            if (e >= E) break;
            float l = a.part[static_cast<size_t>(t) * E + e];
            for (int q = 1; q < KS; ++q) l += a.part[(static_cast<size_t>(q) * a.T + t) * E + e];
            float nw2 = 0.f;
            for (int q = 0; q < KS; ++q) nw2 += a.wsq[(static_cast<size_t>(tt) * KS + q) * E + e];
            const float bl = gam * nx * (sqrtf(nw2) * infl) + 1e-30f;
            const float s = 1.f / (1.f + expf(-l));
            const float sel = s + a.bias[e];
            const float al = fabsf(l);
            const float D = (al > bl) ? fminf(0.25f, expf(-(al - bl)) * 1.01f) : 0.25f;
            w_sel[e] = sel;
            w_bnd[e] = bl * D + 4.f * kU + fabsf(sel) * (2.f * kU);
            w_sc[e] = s;
        }
        __syncwarp();

        // top-K by (sel desc, index asc)
        uint32_t taken = 0;
        float lower_min = FLT_MAX;
        bool order_ok = true;
        float prev_lo = 0.f;
        for (int j = 0; j < K; ++j) {
            float bs = -FLT_MAX;
            int be = INT_MAX;
            for (int i = 0; i < NI; ++i) {
                const int e = lane + 32 * i;
                if (e >= E) break;
                if (taken & (1u << i)) continue;
                const float v = w_sel[e];
                if (be == INT_MAX || before(v, e, bs, be)) { bs = v; be = e; }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float os = __shfl_xor_sync(kFullMask, bs, off);
                const int oe = __shfl_xor_sync(kFullMask, be, off);
                if (oe != INT_MAX && (be == INT_MAX || before(os, oe, bs, be))) { bs = os; be = oe; }
            }
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
            if (lane == 0) w_ord[j] = be;
            const float bb = w_bnd[be];
            const float lo = __fsub_rd(bs, bb), hi = __fadd_ru(bs, bb);
            if (j > 0 && !(prev_lo > hi)) order_ok = false;
            prev_lo = lo;
            lower_min = fminf(lower_min, lo);
        }
        // candidates: every expert whose upper bound reaches the k-th lower bound
        int n_cand = 0;
        uint32_t cand = 0;
        for (int i = 0; i < NI; ++i) {
            const int e = lane + 32 * i;
            const bool c = e < E && __fadd_ru(w_sel[e], w_bnd[e]) >= lower_min;
            if (c) cand |= 1u << i;
            n_cand += __popc(__ballot_sync(kFullMask, c));
        }
        __syncwarp();

        int32_t *oi = a.topk_idx + static_cast<size_t>(t) * K;
        float *ow = a.topk_w + static_cast<size_t>(t) * K;
        if (n_cand == K && order_ok) {
            float den = 0.f;
            for (int j = 0; j < K; ++j) den += w_sc[w_ord[j]];
            for (int j = lane; j < K; j += 32) {
                oi[j] = w_ord[j];
                ow[j] = w_sc[w_ord[j]] / den;
            }
            __syncwarp();
            continue;
        }

        // refine the candidates in double-word arithmetic
        const uint16_t *xrow_p = a.X + static_cast<size_t>(t) * a.H;
        for (int i = 0; i < NI; ++i) {
            uint32_t m = __ballot_sync(kFullMask, (cand >> i) & 1u);
            while (m) {
                const int src = __ffs(m) - 1;
                m &= m - 1;
                const int e = src + 32 * i;
                const double l64 = dot_double_word(xrow_p, a.Wg + static_cast<size_t>(e) * a.H, a.H, lane);
                const double s64 = 1.0 / (1.0 + exp(-l64));
                if (lane == src) w_s64[e] = s64 + static_cast<double>(a.bias[e]);
            }
        }
        __syncwarp();
        uint32_t taken2 = 0;
        for (int j = 0; j < K; ++j) {
            double bs = -DBL_MAX;
            int be = INT_MAX;
            for (int i = 0; i < NI; ++i) {
                if (!((cand >> i) & 1u) || ((taken2 >> i) & 1u)) continue;
                const int e = lane + 32 * i;
                const double v = w_s64[e];
                if (be == INT_MAX || before64(v, e, bs, be)) { bs = v; be = e; }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const double os = __shfl_xor_sync(kFullMask, bs, off);
                const int oe = __shfl_xor_sync(kFullMask, be, off);
                if (oe != INT_MAX && (be == INT_MAX || before64(os, oe, bs, be))) { bs = os; be = oe; }
            }
            if ((be & 31) == lane) taken2 |= 1u << (be >> 5);
            if (lane == 0) w_ord[j] = be;
        }
        __syncwarp();
        double den = 0.0;
        for (int j = 0; j < K; ++j) den += w_s64[w_ord[j]] - static_cast<double>(a.bias[w_ord[j]]);
        for (int j = lane; j < K; j += 32) {
            const int e = w_ord[j];
            oi[j] = e;
            ow[j] = static_cast<float>((w_s64[e] - static_cast<double>(a.bias[e])) / den);
        }
        __syncwarp();
    }
}

}  // namespace

RouterPlan router_plan(int T, int H, int E)
{
    RouterPlan p{};
    p.TT = TT;
    p.TE = TE;
    p.nTT = (T + TT - 1) / TT;
    p.nET = (E + TE - 1) / TE;
    p.S = H / KST;
    const int base = p.nTT * p.nET;
    const int target = 2 * num_sms();
    p.KS = 1;
    while (p.KS * 2 <= p.S && p.KS < 16 && base * p.KS < target) p.KS *= 2;
    auto al = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    p.part_bytes = al(static_cast<size_t>(p.KS) * T * E * sizeof(float));
    p.xsq_bytes = al(static_cast<size_t>(p.KS) * T * sizeof(float));
    p.wsq_bytes = al(static_cast<size_t>(p.nTT) * p.KS * E * sizeof(float));
    p.cnt_bytes = al(static_cast<size_t>(p.nTT) * sizeof(unsigned));
    const size_t gemm_smem = 2 * KST * (TT + TE) * sizeof(float);
    const size_t fin_smem = static_cast<size_t>(NW) * E * (3 * sizeof(float) + sizeof(double)) +
                            NW * 32 * sizeof(int);
    p.smem_bytes = gemm_smem > fin_smem ? gemm_smem : fin_smem;
    return p;
}

cudaError_t launch_router(const void *X, const void *Wg, const float *bias, int T, int H,
                          int E, int K, int32_t *topk_idx, float *topk_w,
                          const RouterPlan &plan, const RouterScratch &scr, int *status,
                          cudaStream_t s)
{
    cudaError_t err = cudaMemsetAsync(scr.cnt, 0, static_cast<size_t>(plan.nTT) * sizeof(unsigned), s);
    if (err != cudaSuccess) return err;
    err = ensure_smem(reinterpret_cast<const void *>(router_kernel), plan.smem_bytes);
    if (err != cudaSuccess) return err;
    RouterArgs a{};
    a.X = static_cast<const uint16_t *>(X);
    a.Wg = static_cast<const uint16_t *>(Wg);
    a.bias = bias;
    a.T = T; a.H = H; a.E = E; a.K = K; a.KS = plan.KS; a.S = plan.S;
    a.part = scr.part; a.xsq = scr.xsq; a.wsq = scr.wsq; a.cnt = scr.cnt;
    a.topk_idx = topk_idx; a.topk_w = topk_w; a.status = status;
    dim3 grid(plan.nET, plan.nTT, plan.KS);
    router_kernel<<<grid, NT, plan.smem_bytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
