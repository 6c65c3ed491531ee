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
// Structure.  Grid (expert tiles, token tiles, K splits).  Each CTA computes a TT x 64
// tile of fp32 logits (TT = 16 tokens for small batches, 64 for large ones) over its slice
// of H on the CUDA cores and writes it to the workspace; the last CTA of a token tile
// (completion counter) sums the split-K partials in a fixed order, scores, selects and
// writes the outputs -- one launch, no host sync.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

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
    int max_pairs;   // capacity of the shared-memory refine list
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

// Double-word accumulation of an exact fp32 product into (hi, lo).
__device__ __forceinline__ void dw_add(float &hi, float &lo, float p)
{
    float s, e;
    two_sum(hi, p, s, e);
    hi = s;
    lo = __fadd_rn(lo, e);
}

// (hi, lo) += (ohi, olo) in double-word arithmetic.
__device__ __forceinline__ void dw_merge(float &hi, float &lo, float ohi, float olo)
{
    float s, e;
    two_sum(hi, ohi, s, e);
    hi = s;
    lo = __fadd_rn(__fadd_rn(lo, olo), e);
}

// Double-word dot product of a bf16 token row and a bf16 gate row, reduced over the warp
// in a fixed order; every lane returns the same value.  Four independent accumulators per
// lane keep four 16-byte loads of each row in flight.
__device__ double dot_double_word(const uint16_t *x, const uint16_t *w, int H, int lane)
{
    const uint4 *xr = reinterpret_cast<const uint4 *>(x);
    const uint4 *wr = reinterpret_cast<const uint4 *>(w);
    const int nv = H / 8;
    float hi[4] = {0.f, 0.f, 0.f, 0.f}, lo[4] = {0.f, 0.f, 0.f, 0.f};
    int v = lane;
    for (; v + 96 < nv; v += 128) {
        uint4 xa[4], wa[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            xa[u] = __ldg(xr + v + 32 * u);
            wa[u] = __ldg(wr + v + 32 * u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float xf[8], wf[8];
            unpack8(xa[u], xf);
            unpack8(wa[u], wf);
#pragma unroll
            for (int i = 0; i < 8; ++i) dw_add(hi[u], lo[u], __fmul_rn(xf[i], wf[i]));  // exact product
        }
    }
    for (; v < nv; v += 32) {
        float xf[8], wf[8];
        unpack8(__ldg(xr + v), xf);
        unpack8(__ldg(wr + v), wf);
#pragma unroll
        for (int i = 0; i < 8; ++i) dw_add(hi[0], lo[0], __fmul_rn(xf[i], wf[i]));
    }
    dw_merge(hi[0], lo[0], hi[1], lo[1]);
    dw_merge(hi[2], lo[2], hi[3], lo[3]);
    dw_merge(hi[0], lo[0], hi[2], lo[2]);
    float h = hi[0], l = lo[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ohi = __shfl_xor_sync(kFullMask, h, off);
        const float olo = __shfl_xor_sync(kFullMask, l, off);
        dw_merge(h, l, ohi, olo);
    }
    return static_cast<double>(h) + static_cast<double>(l);
}

// Top-K of a token among `n` candidate (expert, sel64) pairs by (sel64 desc, expert asc);
// writes the experts and their renormalised weights.  Warp-wide; pairs live in shared memory.
__device__ void select_refined(const int *pe, const double *pv, int n, int K,
                               const float *bias, int32_t *oi, float *ow, int *ord, int lane)
{
    for (int j = 0; j < K; ++j) {
        double bs = -DBL_MAX;
        int be = INT_MAX, bp = -1;
        for (int q = lane; q < n; q += 32) {
            const int e = pe[q];
            if (e < 0) continue;                 // already taken
            const double v = pv[q];
            if (be == INT_MAX || before64(v, e, bs, be)) { bs = v; be = e; bp = q; }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const double os = __shfl_xor_sync(kFullMask, bs, off);
            const int oe = __shfl_xor_sync(kFullMask, be, off);
            const int op = __shfl_xor_sync(kFullMask, bp, off);
            if (oe != INT_MAX && (be == INT_MAX || before64(os, oe, bs, be))) { bs = os; be = oe; bp = op; }
        }
        if (lane == 0) ord[j] = bp;
        __syncwarp();
        if (lane == (bp & 31)) const_cast<int *>(pe)[bp] = -1 - be;   // mark taken, keep expert
        __syncwarp();
    }
    double den = 0.0;
    for (int j = 0; j < K; ++j) {
        const int q = ord[j], e = -1 - pe[q];
        den += pv[q] - static_cast<double>(bias[e]);
    }
    for (int j = lane; j < K; j += 32) {
        const int q = ord[j], e = -1 - pe[q];
        oi[j] = e;
        ow[j] = static_cast<float>((pv[q] - static_cast<double>(bias[e])) / den);
    }
    __syncwarp();
}

template <int TT>
__global__ void __launch_bounds__(NT, 2) router_kernel(const RouterArgs a)
{
    constexpr int TPT = TT / 16;                   // tokens per thread in the tile GEMM
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

    // loaders: X tile = TT rows x 4 vectors of 8 bf16, W tile = 64 rows x 4 vectors
    const bool xload = tid < TT * 4;
    const int xr_row = tid % TT, xr_vec = tid / TT;
    const int wr_row = tid & 63, wr_vec = tid >> 6;
    const int xrow = t0 + xr_row, wrow = e0 + wr_row;
    const bool xok = xload && xrow < a.T, wok = wrow < a.E;
    const uint4 *xp = reinterpret_cast<const uint4 *>(a.X + static_cast<size_t>(xok ? xrow : 0) * a.H) + xr_vec;
    const uint4 *wp = reinterpret_cast<const uint4 *>(a.Wg + static_cast<size_t>(wok ? wrow : 0) * a.H) + wr_vec;
    float xsq = 0.f, wsq = 0.f;
    uint4 xr = make_uint4(0, 0, 0, 0), wr = make_uint4(0, 0, 0, 0);

    const int tx = tid & 15, ty = tid >> 4;        // compute: experts 4tx.., tokens TPT*ty..
    float acc_mid[TPT * 4], acc_out[TPT * 4];
#pragma unroll
    for (int p = 0; p < TPT * 4; ++p) { acc_mid[p] = 0.f; acc_out[p] = 0.f; }

    auto gload = [&](int s) {
        xr = xok ? __ldg(xp + s * 4) : make_uint4(0, 0, 0, 0);
        wr = wok ? __ldg(wp + s * 4) : make_uint4(0, 0, 0, 0);
    };
    auto sstore = [&](int buf) {
        float xf[8], wf[8];
        unpack8(xr, xf);
        unpack8(wr, wf);
        float *wd = wsm + buf * KST * TE + (wr_vec * 8) * TE + wr_row;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            wd[i * TE] = wf[i];
            wsq = fmaf(wf[i], wf[i], wsq);
        }
        if (xload) {
            float *xd = xs + buf * KST * TT + (xr_vec * 8) * TT + xr_row;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                xd[i * TT] = xf[i];
                xsq = fmaf(xf[i], xf[i], xsq);
            }
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
        float acc_in[TPT * 4];
#pragma unroll
        for (int p = 0; p < TPT * 4; ++p) acc_in[p] = 0.f;
        const float *xb = xs + buf * KST * TT + TPT * ty;
        const float *wb = wsm + buf * KST * TE + 4 * tx;
#pragma unroll 8
        for (int kk = 0; kk < KST; ++kk) {
            float xa[TPT];
            if constexpr (TPT == 4) {
                const float4 xv = *reinterpret_cast<const float4 *>(xb + kk * TT);
                xa[0] = xv.x; xa[1] = xv.y; xa[2] = xv.z; xa[3] = xv.w;
            } else {
                xa[0] = xb[kk * TT];
            }
            const float4 wv = *reinterpret_cast<const float4 *>(wb + kk * TE);
            const float wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int i = 0; i < TPT; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc_in[i * 4 + j] = fmaf(xa[i], wa[j], acc_in[i * 4 + j]);
        }
#pragma unroll
        for (int p = 0; p < TPT * 4; ++p) acc_mid[p] += acc_in[p];
        if (++nmid == 8) {
#pragma unroll
            for (int p = 0; p < TPT * 4; ++p) { acc_out[p] += acc_mid[p]; acc_mid[p] = 0.f; }
            nmid = 0;
        }
        if (s + 1 < s_end) sstore(buf ^ 1);
        __syncthreads();
        buf ^= 1;
    }
#pragma unroll
    for (int p = 0; p < TPT * 4; ++p) acc_out[p] += acc_mid[p];

#pragma unroll
    for (int i = 0; i < TPT; ++i) {
        const int t = t0 + TPT * ty + i;
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
        float *rx = xs;            // [4][TT]
        float *rw = xs + 4 * TT;   // [4][64]
        if (xload) rx[xr_vec * TT + xr_row] = xsq;
        rw[wr_vec * 64 + wr_row] = wsq;
        __syncthreads();
        if (tid < TT) {
            const float sx = ((rx[tid] + rx[TT + tid]) + rx[2 * TT + tid]) + rx[3 * TT + tid];
            if (et == 0 && t0 + tid < a.T) a.xsq[static_cast<size_t>(ks) * a.T + t0 + tid] = sx;
        }
        if (tid < 64) {
            const float sw = ((rw[tid] + rw[64 + tid]) + rw[128 + tid]) + rw[192 + tid];
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
    // depth of the summation tree (see the file comment) and the norm inflation
    const int ns_max = (a.S + KS - 1) / KS;
    const float depth = static_cast<float>(KST + 8 + (ns_max + 7) / 8 + 1 + KS + 2);
    const float gam = depth * kU / (1.f - depth * kU) * 1.0001f;
    const float infl = 1.f + static_cast<float>(a.H + 16 + KS) * (2.f * kU) + 4.f * kU;

    // shared: nw[E] | per warp sel[E], bnd[E], sc[E] | per warp ord[32] | pair list
    // (expert, sel64) of the tokens to refine | per warp sel64 scratch for overflow
    float *nw = reinterpret_cast<float *>(smem);
    float *w_sel = nw + E + static_cast<size_t>(warp) * 3 * E;
    float *w_bnd = w_sel + E;
    float *w_sc = w_bnd + E;
    int *w_ord = reinterpret_cast<int *>(nw + E + static_cast<size_t>(NW) * 3 * E) + warp * 32;
    int *p_e = reinterpret_cast<int *>(nw + E + static_cast<size_t>(NW) * 3 * E) + NW * 32;
    int *p_tok = p_e + a.max_pairs;
    unsigned char *after_i = reinterpret_cast<unsigned char *>(p_tok + a.max_pairs);
    after_i = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(after_i) + 7) & ~static_cast<uintptr_t>(7));
    double *p_val = reinterpret_cast<double *>(after_i);
    double *w_s64 = p_val + a.max_pairs + static_cast<size_t>(warp) * E;   // overflow only
    __shared__ int s_npairs, s_npend;
    __shared__ int s_pend[3 * 64];      // (token, first pair, pair count) per pending token
    if (tid == 0) { s_npairs = 0; s_npend = 0; }

    // gate-row norms once per CTA (the K-split partial sums, added in order)
    for (int e = tid; e < E; e += NT) {
        float nw2 = 0.f;
        for (int q = 0; q < KS; ++q) nw2 += a.wsq[(static_cast<size_t>(tt) * KS + q) * E + e];
        nw[e] = sqrtf(nw2) * infl;
    }
    __syncthreads();

    for (int tl = warp; tl < TT; tl += NW) {
        const int t = t0 + tl;
        if (t >= a.T) break;
        float nx2 = 0.f;
        for (int q = 0; q < KS; ++q) nx2 += a.xsq[static_cast<size_t>(q) * a.T + t];
        const float nx = sqrtf(nx2) * infl;

        auto score = [&](int e, float l) {
            const float bl = gam * nx * nw[e] + 1e-30f;
            const float s = 1.f / (1.f + expf(-l));
            const float sel = s + a.bias[e];
            const float al = fabsf(l);
            const float D = (al > bl) ? fminf(0.25f, expf(-(al - bl)) * 1.01f) : 0.25f;
            w_sel[e] = sel;
            w_bnd[e] = bl * D + 4.f * kU + fabsf(sel) * (2.f * kU);
            w_sc[e] = s;
        };
        if ((E & 3) == 0) {
            // coalesced float4 reads of the K-split partials, all issued before the sum
            for (int g = lane; g < E / 4; g += 32) {
                float4 v[16];
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    if (q < KS)
                        v[q] = __ldcg(reinterpret_cast<const float4 *>(
                                   a.part + (static_cast<size_t>(q) * a.T + t) * E) + g);
                float4 l = v[0];
#pragma unroll
                for (int q = 1; q < 16; ++q)
                    if (q < KS) { l.x += v[q].x; l.y += v[q].y; l.z += v[q].z; l.w += v[q].w; }
                score(4 * g, l.x);
                score(4 * g + 1, l.y);
                score(4 * g + 2, l.z);
                score(4 * g + 3, l.w);
            }
        } else {
            for (int e = lane; e < E; e += 32) {
                float l = __ldcg(a.part + static_cast<size_t>(t) * E + e);
                for (int q = 1; q < KS; ++q) l += __ldcg(a.part + (static_cast<size_t>(q) * a.T + t) * E + e);
                score(e, l);
            }
        }
        __syncwarp();

        // top-K by (sel desc, index asc); lane owns experts lane + 32 i
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

        // not certified: queue the candidates for the CTA-wide double-word refine
        int base = 0;
        if (lane == 0) base = atomicAdd(&s_npairs, n_cand);
        base = __shfl_sync(kFullMask, base, 0);
        if (base + n_cand <= a.max_pairs) {
            int pos = base;
            for (int i = 0; i < NI; ++i) {
                const bool c = (cand >> i) & 1u;
                const uint32_t m = __ballot_sync(kFullMask, c);
                if (c) {
                    const int q = pos + __popc(m & ((1u << lane) - 1u));
                    p_e[q] = lane + 32 * i;
                    p_tok[q] = tl;
                }
                pos += __popc(m);
            }
            if (lane == 0) {
                const int pi = atomicAdd(&s_npend, 1);
                s_pend[3 * pi] = tl;
                s_pend[3 * pi + 1] = base;
                s_pend[3 * pi + 2] = n_cand;
            }
            __syncwarp();
            continue;
        }
        // list full (pathological ties): retire the reserved in-range slots, then refine
        // this token with the warp alone
        for (int q = base + lane; q < a.max_pairs; q += 32) p_e[q] = -1;
        const uint16_t *xrow_p = a.X + static_cast<size_t>(t) * a.H;
        int nc = 0;
        int *ce = reinterpret_cast<int *>(w_bnd);      // reuse: candidate experts
        for (int i = 0; i < NI; ++i) {
            const bool c = (cand >> i) & 1u;
            const uint32_t m = __ballot_sync(kFullMask, c);
            if (c) ce[nc + __popc(m & ((1u << lane) - 1u))] = lane + 32 * i;
            nc += __popc(m);
        }
        __syncwarp();
        for (int q = 0; q < nc; ++q) {
            const int e = ce[q];
            const double l64 = dot_double_word(xrow_p, a.Wg + static_cast<size_t>(e) * a.H, a.H, lane);
            if (lane == 0) w_s64[q] = 1.0 / (1.0 + exp(-l64)) + static_cast<double>(a.bias[e]);
        }
        __syncwarp();
        select_refined(ce, w_s64, nc, K, a.bias, oi, ow, w_ord, lane);
    }
    __syncthreads();

    // CTA-wide refine: every warp takes (token, expert) pairs of the queued tokens
    const int npairs = min(s_npairs, a.max_pairs);
    for (int q = warp; q < npairs; q += NW) {
        const int e = p_e[q];
        if (e < 0) continue;
        const int t = t0 + p_tok[q];
        const double l64 = dot_double_word(a.X + static_cast<size_t>(t) * a.H,
                                           a.Wg + static_cast<size_t>(e) * a.H, a.H, lane);
        if (lane == 0) p_val[q] = 1.0 / (1.0 + exp(-l64)) + static_cast<double>(a.bias[e]);
    }
    __syncthreads();
    for (int pi = warp; pi < s_npend; pi += NW) {
        const int tl = s_pend[3 * pi], first = s_pend[3 * pi + 1], cnt = s_pend[3 * pi + 2];
        const int t = t0 + tl;
        select_refined(p_e + first, p_val + first, cnt, K, a.bias,
                       a.topk_idx + static_cast<size_t>(t) * K, a.topk_w + static_cast<size_t>(t) * K,
                       w_ord, lane);
    }
}

}  // namespace

RouterPlan router_plan(int T, int H, int E)
{
    RouterPlan p{};
    p.TT = T <= 4096 ? 16 : 64;
    p.TE = TE;
    p.nTT = (T + p.TT - 1) / p.TT;
    p.nET = (E + TE - 1) / TE;
    p.S = H / KST;
    const int base = p.nTT * p.nET;
    const int target = 2 * num_sms();
    p.KS = 1;
    while (p.KS * 2 <= p.S && p.KS < 8 && base * p.KS < target) p.KS *= 2;
    auto al = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    p.part_bytes = al(static_cast<size_t>(p.KS) * T * E * sizeof(float));
    p.xsq_bytes = al(static_cast<size_t>(p.KS) * T * sizeof(float));
    p.wsq_bytes = al(static_cast<size_t>(p.nTT) * p.KS * E * sizeof(float));
    p.cnt_bytes = al(static_cast<size_t>(p.nTT) * sizeof(unsigned));
    const size_t gemm_smem = 2 * KST * (p.TT + TE) * sizeof(float);
    p.max_pairs = 1024;
    const size_t fin_smem = static_cast<size_t>(E) * sizeof(float) +
                            static_cast<size_t>(NW) * 3 * E * sizeof(float) +
                            NW * 32 * sizeof(int) + 2 * p.max_pairs * sizeof(int) + 16 +
                            p.max_pairs * sizeof(double) +
                            static_cast<size_t>(NW) * E * sizeof(double);
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
    const void *fn = plan.TT == 16 ? reinterpret_cast<const void *>(router_kernel<16>)
                                   : reinterpret_cast<const void *>(router_kernel<64>);
    err = ensure_smem(fn, plan.smem_bytes);
    if (err != cudaSuccess) return err;
    RouterArgs a{};
    a.X = static_cast<const uint16_t *>(X);
    a.Wg = static_cast<const uint16_t *>(Wg);
    a.bias = bias;
    a.T = T; a.H = H; a.E = E; a.K = K; a.KS = plan.KS; a.S = plan.S;
    a.part = scr.part; a.xsq = scr.xsq; a.wsq = scr.wsq; a.cnt = scr.cnt;
    a.topk_idx = topk_idx; a.topk_w = topk_w; a.status = status;
    a.max_pairs = plan.max_pairs;
    dim3 grid(plan.nET, plan.nTT, plan.KS);
    if (plan.TT == 16)
        router_kernel<16><<<grid, NT, plan.smem_bytes, s>>>(a);
    else
        router_kernel<64><<<grid, NT, plan.smem_bytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
