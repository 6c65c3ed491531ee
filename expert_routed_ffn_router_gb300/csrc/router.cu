// router.cu -- fused MoE router: gate GEMM -> sigmoid scoring -> selection bias -> top-k
// -> renormalised weights.
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
// summation is a fixed tree in which every product passes through at most
//     d = 32 (one 32-deep chain per shared-memory stage) + stages per split + splits + 2
// additions, so |l_fp32 - l| <= gamma_d * sum|x_h w_h| <= gamma_d * ||x|| * ||w||
// (Cauchy-Schwarz), gamma_d = d u / (1 - d u), u = 2^-24.  Propagating that bound through
// the sigmoid and the bias add gives an interval per expert.  When the intervals certify
// both the chosen set and its order, the fp32 result is exact; otherwise the candidates
// are the experts whose interval reaches the k-th lower bound, and those whose interval
// meets another candidate's (every candidate, under the other routing options) are
// re-scored in double-word fp32 arithmetic (error-free TwoSum accumulation of the exact
// products, ~2^-48 relative) with an fp64 sigmoid; the top-k is taken again among the
// candidates (the others keep their fp32 sel, which orders exactly since their intervals
// are disjoint from every other candidate's).
//
// Structure.  A grid (expert tiles, token tiles, K splits) of CTAs (256 threads; 384 for
// the warp-specialised tiles) computes fp32 logit tiles on the CUDA cores:
//   tiny batches (T <= 8):       four warps per expert, all tokens at once;
//   9 to 15 and 2049 to 4096:    16 tokens x 256 experts per CTA, 4x4 per thread;
//   16 to 2048 tokens:           16 tokens x 256 experts per CTA, 4x4 per thread on eight
//                                compute warps, fed through a 4-stage fp32 ring by four
//                                producer warps (cp.async staging, bf16 -> fp32, norms);
//   large batches (T > 4096):    128 tokens x 128 experts per CTA, 8x8 per thread, the
//                                same warp-specialised structure.
// Up to 15 tokens and from 2049 to 4096 tokens the last CTA of a token tile (completion
// counter) sums the split-K partials in a fixed order, scores, selects and writes the
// outputs -- one launch.  From 16 to 2048 tokens and for large batches a second launch
// finalises 1 to 8 tokens a CTA (split-K sum, scoring and certified top-K, then the
// CTA-wide re-score of the uncertified candidates), so the selection is spread over the
// whole GPU instead of one CTA per token tile.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int KST = 32;    // k per shared-memory stage
constexpr int NT = 256;    // threads
constexpr int NW = NT / 32;
constexpr int CH = 16;     // tokens per finalise chunk (two per warp)
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
    int depth;       // additions any product passes through in its logit's summation
    // routing options (all at their defaults: sigmoid, one group, renormalised weights)
    int scoring;     // 0 sigmoid, 1 softmax over the token's E logits
    int n_group;     // groups of E / n_group consecutive experts (<= 32)
    int topk_group;  // groups kept per token
    int group_top;   // a group's score: the sum of its group_top (1 or 2) largest sel
    int renorm;      // 1: weights = selected s / their sum; 0: the selected s
    int variant;     // any option off its default: the general selection path
};

// Two-stage CTA tile (gemm_tile): TT tokens x TE experts, TPT x EPT per thread, PF stages
// of loads in flight in registers.
template <int TT_, int TE_, int TPT_, int EPT_, int PF_>
struct Cfg {
    static constexpr int TT = TT_, TE = TE_, TPT = TPT_, EPT = EPT_, PF = PF_;
    static constexpr int NTY = TT / TPT, NTX = TE / EPT;
    static constexpr int LY = 4;                          // token groups per warp
    static constexpr int XV = TT * 4, WV = TE * 4;        // 8-element vectors per stage
    static constexpr int XPT = (XV + NT - 1) / NT, WPT = (WV + NT - 1) / NT;
    static_assert(NTX * NTY == NT, "one output micro-tile per thread");
    static_assert(NTY % LY == 0 && NTX % (32 / LY) == 0, "warp layout");
    static_assert(EPT == 4 && TPT % 4 == 0, "float4 operand reads");
};
using SmallCfg = Cfg<16, 256, 4, 4, 2>;

// Warp-specialised CTA tile (gemm_tile_ws): TT x TE on the eight compute warps, TPT x EPT
// outputs a thread in paired fp32 FMAs (two tokens per instruction -- the same correctly
// rounded operations in the same order as two fmaf, in half the FMA instructions).
template <int TT_, int TE_, int TPT_, int EPT_, int RING_ = 4, int STG_ = 4>
struct WsCfg {
    static constexpr int TT = TT_, TE = TE_, TPT = TPT_, EPT = EPT_;
    static constexpr int RING = RING_, STG = STG_;        // fp32 ring and bf16 staging stages
    static constexpr int NTY = TT / TPT, NTX = TE / EPT;
    static constexpr int LY = 4;                          // token groups per warp
    static_assert(NTX * NTY == NT, "one output micro-tile per compute thread");
    static_assert(NTY % LY == 0 && NTX % (32 / LY) == 0, "warp layout");
    static_assert(EPT % 4 == 0 && TPT % 4 == 0, "float4 operand reads");
};
// 8 x 8 outputs a thread: 16 operands read from shared memory per 64 FMAs (the 8 x 4 tile
// read 12 per 32 and was bound by shared-memory bandwidth); one CTA per SM holds the
// 64 paired running sums.
using LargeCfg = WsCfg<128, 128, 8, 8>;
// 16 tokens x 256 experts, 4 x 4 outputs a thread, for batches of 16 to 2048 tokens: one
// CTA per SM (four-stage fp32 and staging rings).
using SmallWsCfg = WsCfg<16, 256, 4, 4, 4, 4>;

// Two fp32 lanes per 64-bit register: d = a * b + c and d = a + b, each lane correctly
// rounded (the same results as two fmaf / two fp32 adds).
__device__ __forceinline__ uint64_t fma_x2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t add_x2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t dup_x2(float w)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(w));
    return d;
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Order of (score, expert): larger score first, then lower expert index.  A NaN score
// (non-finite inputs) orders below every number, so the order stays total and the lanes of
// a warp reduction agree on its winner.
__device__ __forceinline__ bool before64(double a, int ea, double b, int eb)
{
    a = a == a ? a : -INFINITY;
    b = b == b ? b : -INFINITY;
    return a > b || (a == b && ea < eb);
}

// Total order key of (sel, e): larger sel first, then lower expert index.
__device__ __forceinline__ unsigned long long rank_key(float sel, int e)
{
    uint32_t u = __float_as_uint(sel + 0.0f);            // -0 -> +0
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);       // monotone float -> uint
    return (static_cast<unsigned long long>(u) << 32) | static_cast<uint32_t>(~e);
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
// in a fixed order; every lane returns the same value.  Eight independent accumulators
// per lane keep eight 16-byte loads of each row in flight.
__device__ double dot_double_word(const uint16_t *x, const uint16_t *w, int H, int lane)
{
    constexpr int U = 8;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x);
    const uint4 *wr = reinterpret_cast<const uint4 *>(w);
    const int nv = H / 8;
    float hi[U], lo[U];
#pragma unroll
    for (int u = 0; u < U; ++u) { hi[u] = 0.f; lo[u] = 0.f; }
    int v = lane;
    for (; v + 32 * (U - 1) < nv; v += 32 * U) {
        uint4 xa[U], wa[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            xa[u] = __ldg(xr + v + 32 * u);
            wa[u] = __ldg(wr + v + 32 * u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float xf[8], wf[8];
            unpack8(xa[u], xf);
            unpack8(wa[u], wf);
#pragma unroll
            for (int i = 0; i < 8; ++i) dw_add(hi[u], lo[u], __fmul_rn(xf[i], wf[i]));  // exact product
        }
    }
    if (v < nv) {                          // tail: one predicated batch of loads
        uint4 xa[U], wa[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool ok = v + 32 * u < nv;
            xa[u] = ok ? __ldg(xr + v + 32 * u) : make_uint4(0, 0, 0, 0);
            wa[u] = ok ? __ldg(wr + v + 32 * u) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float xf[8], wf[8];
            unpack8(xa[u], xf);
            unpack8(wa[u], wf);
#pragma unroll
            for (int i = 0; i < 8; ++i) dw_add(hi[u], lo[u], __fmul_rn(xf[i], wf[i]));
        }
    }
#pragma unroll
    for (int step = 1; step < U; step <<= 1)
#pragma unroll
        for (int u = 0; u + step < U; u += 2 * step) dw_merge(hi[u], lo[u], hi[u + step], lo[u + step]);
    float h = hi[0], l = lo[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ohi = __shfl_xor_sync(kFullMask, h, off);
        const float olo = __shfl_xor_sync(kFullMask, l, off);
        dw_merge(h, l, ohi, olo);
    }
    return static_cast<double>(h) + static_cast<double>(l);
}

// Monotone 64-bit key of an fp64 score: a larger score gives a larger key; -0 and +0 give
// the same key; NaN gives the key of -infinity (it orders below every number).
__device__ __forceinline__ unsigned long long key64(double v)
{
    v = v == v ? v + 0.0 : -INFINITY;
    const unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(v));
    return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

// Top-K of a token among `n` candidate (expert, sel64) pairs by (sel64 desc, expert asc);
// writes the experts and their renormalised weights.  Warp-wide; pairs live in shared
// memory; taken pairs are marked by storing -1 - expert.  The order is the one before64
// defines, decided on integer keys: every lane keeps its best untaken pair as (key64 of
// the score, ~expert), and a round's winner is the lane maximum of the score keys, then of
// ~expert among the lanes that hold that key (hardware reductions, no fp64 compares).
__device__ void select_refined(int *pe, const double *pv, int n, int K, const float *bias,
                               int32_t *oi, float *ow, int *ord, int lane, int renorm = 1)
{
    // lists of up to 32 candidates (the usual case): each lane's key in registers
    const bool reg = n <= 32;
    const unsigned long long rk = (reg && lane < n) ? key64(pv[lane]) : 0ull;
    for (int j = 0; j < K; ++j) {
        unsigned long long bk = 0ull;     // 0: no untaken pair (every real key is larger)
        uint32_t bi = 0u;                 // ~expert of the lane's best
        int bp = -1;
        if (reg) {
            if (lane < n && pe[lane] >= 0) { bk = rk; bi = ~static_cast<uint32_t>(pe[lane]); bp = lane; }
        } else {
            for (int q = lane; q < n; q += 32) {
                const int e = pe[q];
                if (e < 0) continue;
                const unsigned long long k = key64(pv[q]);
                const uint32_t ie = ~static_cast<uint32_t>(e);
                if (k > bk || (k == bk && ie > bi)) { bk = k; bi = ie; bp = q; }
            }
        }
        const uint32_t kh = static_cast<uint32_t>(bk >> 32), kl = static_cast<uint32_t>(bk);
        const uint32_t mh = __reduce_max_sync(kFullMask, kh);
        const uint32_t ml = __reduce_max_sync(kFullMask, kh == mh ? kl : 0u);
        const bool top = kh == mh && kl == ml;
        const uint32_t mi = __reduce_max_sync(kFullMask, top ? bi : 0u);
        const uint32_t win = __ballot_sync(kFullMask, top && bi == mi && bp >= 0);
        const int wp = win ? __shfl_sync(kFullMask, bp, __ffs(win) - 1) : -1;
        if (lane == 0) ord[j] = wp;
        __syncwarp();
        if (wp >= 0 && lane == (wp & 31)) pe[wp] = -1 - pe[wp];
        __syncwarp();
    }
    // weights: the selected unbiased scores (fp64 minus the bias), renormalised in fp32
    // (a relative error of a few 1e-7); lane j < K holds slot j.  A round that found no
    // pair (callers pass at least K candidates) writes expert 0 with weight 0 rather than
    // an index outside the list.
    int e = 0;
    float sc = 0.f;
    const int q = lane < K ? ord[lane] : -1;
    if (q >= 0) {
        e = pe[q] < 0 ? -1 - pe[q] : pe[q];
        sc = static_cast<float>(pv[q] - static_cast<double>(bias[e]));
    }
    float den = 0.f;
    for (int j = 0; j < K; ++j) den += __shfl_sync(kFullMask, sc, j);
    if (lane < K) {
        oi[lane] = e;
        ow[lane] = q < 0 ? 0.f : (renorm ? sc / den : sc);
    }
    __syncwarp();
}

// Double-word partial dot product of a token row and a gate row over the 8-element
// vectors [v0, v1), reduced over the warp in a fixed order (every lane gets (h, l)).  A
// group of warps splits one dot into such ranges and merges the partials in rank order.
__device__ void dot_dw_range(const uint16_t *x, const uint16_t *w, int v0, int v1, int lane,
                             float &h, float &l)
{
    constexpr int U = 8;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x);
    const uint4 *wr = reinterpret_cast<const uint4 *>(w);
    float hi[U], lo[U];
#pragma unroll
    for (int u = 0; u < U; ++u) { hi[u] = 0.f; lo[u] = 0.f; }
    for (int v = v0 + lane; v < v1; v += 32 * U) {
        uint4 xa[U], wa[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool ok = v + 32 * u < v1;
            xa[u] = ok ? __ldg(xr + v + 32 * u) : make_uint4(0, 0, 0, 0);
            wa[u] = ok ? __ldg(wr + v + 32 * u) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float xf[8], wf[8];
            unpack8(xa[u], xf);
            unpack8(wa[u], wf);
#pragma unroll
            for (int i = 0; i < 8; ++i) dw_add(hi[u], lo[u], __fmul_rn(xf[i], wf[i]));  // exact product
        }
    }
#pragma unroll
    for (int step = 1; step < U; step <<= 1)
#pragma unroll
        for (int u = 0; u + step < U; u += 2 * step) dw_merge(hi[u], lo[u], hi[u + step], lo[u + step]);
    h = hi[0];
    l = lo[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ohi = __shfl_xor_sync(kFullMask, h, off);
        const float olo = __shfl_xor_sync(kFullMask, l, off);
        dw_merge(h, l, ohi, olo);
    }
}

// Bound constants of the summation tree: gamma_d and the inflation of computed norms.
struct Bounds {
    float gam, infl;
    __device__ Bounds(int depth, int KS, int H)
    {
        const float d = static_cast<float>(depth);
        gam = d * kU / (1.f - d * kU) * 1.0001f;
        infl = 1.f + static_cast<float>(H + 16 + KS) * (2.f * kU) + 4.f * kU;
    }
};

// Warp-wide maximum of 64-bit keys: the high words' maximum, then the low words' maximum
// among the lanes holding it (two hardware reductions instead of five 64-bit shuffles).
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v)
{
    const uint32_t hi = static_cast<uint32_t>(v >> 32), lo = static_cast<uint32_t>(v);
    const uint32_t mh = __reduce_max_sync(kFullMask, hi);
    const uint32_t ml = __reduce_max_sync(kFullMask, hi == mh ? lo : 0u);
    return (static_cast<unsigned long long>(mh) << 32) | ml;
}

// Compare-and-swap for a descending order of 64-bit keys.
__device__ __forceinline__ void cas_desc(unsigned long long &a, unsigned long long &b)
{
    const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
    a = hi;
    b = lo;
}

// Sorts eight keys in descending order (Batcher's odd-even merge network, 19 comparators).
__device__ __forceinline__ void sort8_desc(unsigned long long (&k)[8])
{
    cas_desc(k[0], k[1]); cas_desc(k[2], k[3]); cas_desc(k[4], k[5]); cas_desc(k[6], k[7]);
    cas_desc(k[0], k[2]); cas_desc(k[1], k[3]); cas_desc(k[4], k[6]); cas_desc(k[5], k[7]);
    cas_desc(k[1], k[2]); cas_desc(k[5], k[6]);
    cas_desc(k[0], k[4]); cas_desc(k[1], k[5]); cas_desc(k[2], k[6]); cas_desc(k[3], k[7]);
    cas_desc(k[2], k[4]); cas_desc(k[3], k[5]);
    cas_desc(k[1], k[2]); cas_desc(k[3], k[4]); cas_desc(k[5], k[6]);
}

// Score, selection key and error bound of one expert of a token: l is the fp32 logit,
// bl = gam ||x|| ||w_e|| bounds its summation error; s = sigmoid(l) and sel = s + b carry
// the bound propagated through the sigmoid (|sigmoid'| <= min(1/4, e^-(|l| - bl))) plus the
// fp32 rounding of the sigmoid and of the add.
__device__ __forceinline__ void score_expert(float l, float bl, float b, float &sel, float &bnd,
                                             float &s)
{
    s = 1.f / (1.f + expf(-l));
    sel = s + b;
    const float al = fabsf(l);
    const float D = (al > bl) ? fminf(0.25f, __expf(-(al - bl)) * 1.01f) : 0.25f;
    bnd = bl * D + 4.f * kU + fabsf(sel) * (2.f * kU);
}

// Selects the top-K of one token held by one warp from its scored experts (w_sel, w_bnd,
// w_sc as score_expert leaves them; lane owns e = lane + 32i) in fp32 with the certified
// error bound.  Returns true when the result is certified and written; otherwise `cand`
// holds the lane's candidate bits and `n_cand` their warp-wide count.
__device__ bool select_scored(int E, int K, const float *w_sel, const float *w_bnd,
                              const float *w_sc, int32_t *oi, float *ow, uint32_t &cand,
                              int &n_cand, int lane)
{
    const int NI = (E + 31) / 32;
    const bool fast = NI <= 8;                // keys of <= 256 experts fit in registers
    unsigned long long key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) key[i] = 0ull;
    unsigned long long best = 0ull;           // generic path: lane's best untaken key
    if (fast) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            if (i < NI && e < E) key[i] = rank_key(w_sel[e], e);
        }
        sort8_desc(key);
    } else {
        for (int i = 0; i < NI; ++i) {
            const int e = lane + 32 * i;
            if (e >= E) break;
            const unsigned long long k = rank_key(w_sel[e], e);
            best = k > best ? k : best;
        }
    }

    uint32_t taken = 0;
    float lower_min = FLT_MAX, prev_lo = 0.f, my_s = 0.f;
    int my_e = 0;
    bool order_ok = true;
    for (int j = 0; j < K; ++j) {
        // tournament over the lanes' heads (fast path: a lane's keys are kept sorted)
        const unsigned long long head = fast ? key[0] : best;
        const unsigned long long win = warp_max_u64(head);
        const int e = static_cast<int>(~static_cast<uint32_t>(win));
        if (fast) {
            if (head == win) {                 // pop the winner's head
#pragma unroll
                for (int u = 0; u < 7; ++u) key[u] = key[u + 1];
                key[7] = 0ull;
            }
        } else if ((e & 31) == lane) {         // generic: the owner rescans its entries
            taken |= 1u << (e >> 5);
            best = 0ull;
            for (int i = 0; i < NI; ++i) {
                const int f = lane + 32 * i;
                if (f >= E) break;
                if (taken & (1u << i)) continue;
                const unsigned long long k = rank_key(w_sel[f], f);
                best = k > best ? k : best;
            }
        }
        const float ws = w_sel[e], wb = w_bnd[e];
        if (lane == j) { my_e = e; my_s = w_sc[e]; }
        const float lo = __fsub_rd(ws, wb), hi = __fadd_ru(ws, wb);
        if (j > 0 && !(prev_lo > hi)) order_ok = false;
        prev_lo = lo;
        lower_min = fminf(lower_min, lo);
    }
    // candidates: every expert whose upper bound reaches the k-th lower bound
    n_cand = 0;
    cand = 0;
    for (int i = 0; i < NI; ++i) {
        const int e = lane + 32 * i;
        const bool c = e < E && __fadd_ru(w_sel[e], w_bnd[e]) >= lower_min;
        if (c) cand |= 1u << i;
        n_cand += __popc(__ballot_sync(kFullMask, c));
    }
    if (n_cand == K && order_ok) {
        float den = 0.f;
        for (int j = 0; j < K; ++j) den += __shfl_sync(kFullMask, my_s, j);
        if (lane < K) {
            oi[lane] = my_e;
            ow[lane] = my_s / den;
        }
        __syncwarp();
        return true;
    }
    __syncwarp();
    return false;
}

// Scores one token held by one warp (`w_sel` holds its fp32 logits on entry and receives
// sel; w_bnd / w_sc receive the bound and the sigmoid) and selects its top-K as
// select_scored does.
__device__ bool score_select(int E, int K, float nx, const float *nw, const float *bias,
                             float gam, float *w_sel, float *w_bnd, float *w_sc,
                             int32_t *oi, float *ow, uint32_t &cand, int &n_cand, int lane)
{
    for (int e = lane; e < E; e += 32) {
        float sel, bnd, sc;
        score_expert(w_sel[e], gam * nx * nw[e] + 1e-30f, bias[e], sel, bnd, sc);
        w_sel[e] = sel;
        w_bnd[e] = bnd;
        w_sc[e] = sc;
    }
    __syncwarp();
    return select_scored(E, K, w_sel, w_bnd, w_sc, oi, ow, cand, n_cand, lane);
}

__device__ __forceinline__ float warp_max_f(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, off));
    return v;
}

__device__ __forceinline__ float warp_min_f(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fminf(v, __shfl_xor_sync(kFullMask, v, off));
    return v;
}


// The largest two of a sequence (v1 >= v2), for a group's score.
__device__ __forceinline__ void top2_push(float v, float &v1, float &v2)
{
    if (v > v1) { v2 = v1; v1 = v; } else if (v > v2) { v2 = v; }
}

// Scores one token with the general routing options (softmax scoring, group-limited
// selection, unnormalised weights) and selects its top-K in fp32 with certified bounds.
// Returns 1 when the result is certified and written.  With sigmoid scores, returns 0
// when it is not: `cand` / `n_cand` hold the experts to re-score and `ck` / `ug` the
// groups certainly kept / still undecided (bit g), for select_candidates64.  The
// candidates are the members of undecided groups that may be among their group's
// group_top best (upper bound >= the group's group_top-th lower bound) and the experts of
// kept or undecided groups whose upper bound reaches the K-th largest lower bound among
// the experts of the certainly kept groups.  With softmax scores returns -1 instead: the
// caller re-scores every expert (the normaliser needs all of them) for select_general64.
//
// Softmax bound.  With every logit within beta of its fp32 value, the exact s_e lies
// within a factor e^{+-2 beta} of exp(l^_e) / sum_j exp(l^_j) (numerator and denominator
// each move by at most e^{+-beta}).  Its fp32 evaluation exp(l^_e - m) / sum adds
// u |l^_e - m| for the subtraction in the exponent, 2 ulp (4u) for expf in numerator and
// every summand, (lane terms + 5 tree levels) u for the positive sum and u for the
// division.  An absolute 1e-30 covers underflowed terms.
//
// Group bound.  A group's score (sum of its n largest sel) is non-decreasing in every sel,
// so the sums of the n largest lower / upper bounds enclose it.  The kept groups are
// certified when the smallest lower bound among them exceeds the largest upper bound of
// the others.
__device__ int score_select_general(const RouterArgs &a, float nx, const float *nw,
                                    const float *bias, float gam, float *w_sel, float *w_bnd,
                                    float *w_sc, int32_t *oi, float *ow, uint32_t &cand,
                                    int &n_cand, uint32_t &ck, uint32_t &ug, int lane)
{
    const int E = a.E, K = a.K, NI = (E + 31) / 32;
    if (a.scoring == 0) {
        for (int i = 0; i < NI; ++i) {
            const int e = lane + 32 * i;
            if (e >= E) break;
            const float l = w_sel[e];
            const float bl = gam * nx * nw[e] + 1e-30f;
            const float s = 1.f / (1.f + expf(-l));
            const float sel = s + bias[e];
            const float al = fabsf(l);
            const float D = (al > bl) ? fminf(0.25f, __expf(-(al - bl)) * 1.01f) : 0.25f;
            w_sel[e] = sel;
            w_bnd[e] = bl * D + 4.f * kU + fabsf(sel) * (2.f * kU);
            w_sc[e] = s;
        }
    } else {
        float m = -FLT_MAX, beta = 0.f;
        for (int i = 0; i < NI; ++i) {
            const int e = lane + 32 * i;
            if (e >= E) break;
            m = fmaxf(m, w_sel[e]);
            beta = fmaxf(beta, gam * nx * nw[e] + 1e-30f);
        }
        m = warp_max_f(m);
        beta = warp_max_f(beta);
        float sum = 0.f, spread = 0.f;
        for (int i = 0; i < NI; ++i) {
            const int e = lane + 32 * i;
            if (e >= E) break;
            const float d = w_sel[e] - m;
            const float A = expf(d);
            w_sc[e] = A;
            sum += A;
            spread = fmaxf(spread, -d);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFullMask, sum, off);
        spread = warp_max_f(spread);
        const float rel = (expm1f(2.f * beta) + kU * (2.f * spread + static_cast<float>(NI) + 14.f)) * 1.02f;
        for (int i = 0; i < NI; ++i) {
            const int e = lane + 32 * i;
            if (e >= E) break;
            const float sc = w_sc[e] / sum;
            const float sel = sc + bias[e];
            w_sc[e] = sc;
            w_sel[e] = sel;
            w_bnd[e] = sc * rel + 1e-30f + fabsf(sel) * (2.f * kU);
        }
    }
    __syncwarp();

    // groups kept (bit g), certified against the others
    uint32_t kmask = kFullMask;
    int G = E;
    bool groups_ok = true;
    float nth_lo = -FLT_MAX;       // lane g: the group_top-th largest lower bound of group g
    ck = kFullMask;
    ug = 0u;
    if (a.n_group > 1) {
        const int ng = a.n_group;
        G = E / ng;
        float glo = -FLT_MAX, ghi = -FLT_MAX;
        unsigned long long key = 0ull;
        float s1 = -FLT_MAX, s2 = -FLT_MAX, l1 = -FLT_MAX, l2 = -FLT_MAX, h1 = -FLT_MAX, h2 = -FLT_MAX;
        if (lane < ng) {
            for (int e = lane * G; e < (lane + 1) * G; ++e) {
                const float v = w_sel[e], b = w_bnd[e];
                top2_push(v, s1, s2);
                top2_push(__fsub_rd(v, b), l1, l2);
                top2_push(__fadd_ru(v, b), h1, h2);
            }
            const bool two = a.group_top == 2;
            key = rank_key(two ? s1 + s2 : s1, lane);
            glo = two ? __fadd_rd(l1, l2) : l1;
            ghi = two ? __fadd_ru(h1, h2) : h1;
        }
        kmask = 0u;
        for (int r = 0; r < a.topk_group; ++r) {
            const unsigned long long win = warp_max_u64(key);
            if (win == 0ull) break;        // (topk_group <= n_group: not reached)
            const int g = static_cast<int>(~static_cast<uint32_t>(win));
            kmask |= 1u << g;
            if (lane == g) key = 0ull;
        }
        const bool kept = lane < ng && ((kmask >> lane) & 1u);
        const float klo = warp_min_f(kept ? glo : FLT_MAX);
        const float ohi = warp_max_f(lane < ng && !kept ? ghi : -FLT_MAX);
        ck = kmask;
        if (a.topk_group < ng && !(klo > ohi)) {
            if (a.scoring != 0) return -1;
            // a kept group above every other group's upper bound is kept for certain, an
            // other group below every kept group's lower bound is dropped for certain
            groups_ok = false;
            ck = __ballot_sync(kFullMask, kept && glo > ohi);
            ug = __ballot_sync(kFullMask, lane < ng && !(kept && glo > ohi) && !(!kept && ghi < klo));
            nth_lo = a.group_top == 2 ? l2 : l1;
        }
    }

    if (!groups_ok) {
        // K-th largest lower bound among the experts of the certainly kept groups
        uint32_t tk = 0;
        auto best_lo = [&]() {
            unsigned long long b = 0ull;
            for (int i = 0; i < NI; ++i) {
                const int e = lane + 32 * i;
                if (e >= E) break;
                if ((tk >> i) & 1u || !((ck >> (e / G)) & 1u)) continue;
                const unsigned long long k = rank_key(__fsub_rd(w_sel[e], w_bnd[e]), e);
                b = k > b ? k : b;
            }
            return b;
        };
        unsigned long long b = best_lo();
        float L = FLT_MAX;
        for (int j = 0; j < K; ++j) {
            const unsigned long long win = warp_max_u64(b);
            if (win == 0ull) { L = -FLT_MAX; break; }     // fewer than K such experts
            const int e = static_cast<int>(~static_cast<uint32_t>(win));
            if ((e & 31) == lane) {
                tk |= 1u << (e >> 5);
                b = best_lo();
            }
            L = fminf(L, __fsub_rd(w_sel[e], w_bnd[e]));
        }
        n_cand = 0;
        cand = 0;
        for (int i = 0; i < NI; ++i) {
            const int e = lane + 32 * i;
            const int g = e < E ? e / G : 0;
            const float gth = __shfl_sync(kFullMask, nth_lo, g);
            bool c = false;
            if (e < E) {
                const float hi = __fadd_ru(w_sel[e], w_bnd[e]);
                const bool live = ((ck | ug) >> g) & 1u;
                c = (live && hi >= L) || (((ug >> g) & 1u) && hi >= gth);
            }
            if (c) cand |= 1u << i;
            n_cand += __popc(__ballot_sync(kFullMask, c));
        }
        __syncwarp();
        return 0;
    }

    // top-K among the experts of the kept groups: each lane keeps its best untaken key
    auto eligible = [&](int e) { return ((kmask >> (e / G)) & 1u) != 0u; };
    uint32_t taken = 0;
    auto lane_best = [&]() {
        unsigned long long b = 0ull;
        for (int i = 0; i < NI; ++i) {
            const int e = lane + 32 * i;
            if (e >= E) break;
            if ((taken >> i) & 1u || !eligible(e)) continue;
            const unsigned long long k = rank_key(w_sel[e], e);
            b = k > b ? k : b;
        }
        return b;
    };
    unsigned long long best = lane_best();
    float lower_min = FLT_MAX, prev_lo = 0.f, my_s = 0.f;
    int my_e = 0;
    bool order_ok = true;
    for (int j = 0; j < K; ++j) {
        const unsigned long long win = warp_max_u64(best);
        const int e = static_cast<int>(~static_cast<uint32_t>(win));
        if ((e & 31) == lane) {
            taken |= 1u << (e >> 5);
            best = lane_best();
        }
        const float ws = w_sel[e], wb = w_bnd[e];
        if (lane == j) { my_e = e; my_s = w_sc[e]; }
        const float lo = __fsub_rd(ws, wb), hi = __fadd_ru(ws, wb);
        if (j > 0 && !(prev_lo > hi)) order_ok = false;
        prev_lo = lo;
        lower_min = fminf(lower_min, lo);
    }
    n_cand = 0;
    cand = 0;
    for (int i = 0; i < NI; ++i) {
        const int e = lane + 32 * i;
        const bool c = e < E && eligible(e) && __fadd_ru(w_sel[e], w_bnd[e]) >= lower_min;
        if (c) cand |= 1u << i;
        n_cand += __popc(__ballot_sync(kFullMask, c));
    }
    if (n_cand != K || !order_ok) {
        __syncwarp();
        return a.scoring == 0 ? 0 : -1;
    }
    float den = 0.f;
    for (int j = 0; j < K; ++j) den += __shfl_sync(kFullMask, my_s, j);
    if (lane < K) {
        oi[lane] = my_e;
        ow[lane] = a.renorm ? my_s / den : my_s;
    }
    __syncwarp();
    return 1;
}

// The selection from re-scored sigmoid candidates (score_select_general's 0 case): pv[q]
// holds the fp64 logit of expert pe[q] on entry and is turned into sel = sigmoid + bias.
// Undecided groups (bit g of ug) are scored by the group_top best sel of their candidates
// -- every member that can be among them is a candidate -- and the best of them join the
// certainly kept groups (ck) up to topk_group (equal scores: lower group first); the top-K
// is then taken among the candidates of the kept groups.
__device__ void select_candidates64(const RouterArgs &a, int *pe, double *pv, int n,
                                    uint32_t ck, uint32_t ug, int32_t *oi, float *ow, int *ord,
                                    int lane)
{
    for (int q = lane; q < n; q += 32)
        pv[q] = 1.0 / (1.0 + exp(-pv[q])) + static_cast<double>(a.bias[pe[q]]);
    __syncwarp();
    const int G = a.E / a.n_group;
    uint32_t kept = ck;
    if (ug) {
        double gs = -DBL_MAX;
        bool in = ((ug >> lane) & 1u) != 0u;
        if (in) {
            double s1 = -DBL_MAX, s2 = -DBL_MAX;
            for (int q = 0; q < n; ++q) {
                if (pe[q] / G != lane) continue;
                const double v = pv[q];
                if (v > s1) { s2 = s1; s1 = v; } else if (v > s2) { s2 = v; }
            }
            gs = a.group_top == 2 ? s1 + s2 : s1;
        }
        const int more = a.topk_group - __popc(ck);
        for (int r = 0; r < more; ++r) {
            double bs = in ? gs : -DBL_MAX;
            int bg = in ? lane : INT_MAX;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const double os = __shfl_xor_sync(kFullMask, bs, off);
                const int og = __shfl_xor_sync(kFullMask, bg, off);
                if (og != INT_MAX && (bg == INT_MAX || before64(os, og, bs, bg))) { bs = os; bg = og; }
            }
            if (bg == INT_MAX) break;      // no undecided group left
            kept |= 1u << bg;
            if (lane == bg) in = false;
        }
    }
    __syncwarp();
    for (int q = lane; q < n; q += 32)
        if (!((kept >> (pe[q] / G)) & 1u)) pe[q] = -1 - pe[q];
    __syncwarp();
    select_refined(pe, pv, n, a.K, a.bias, oi, ow, ord, lane, a.renorm);
}

// The general routing options in fp64 from re-scored logits of EVERY expert of a token:
// pv[e] holds expert e's logit on entry (pe[e] == e); pv is overwritten with the scores,
// pe marks taken experts as -1 - e.  Warp-wide.
__device__ void select_general64(const RouterArgs &a, int *pe, double *pv, int32_t *oi,
                                 float *ow, int *ord, int lane)
{
    const int E = a.E, K = a.K;
    if (a.scoring == 1) {
        double m = -DBL_MAX;
        for (int e = lane; e < E; e += 32) m = fmax(m, pv[e]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmax(m, __shfl_xor_sync(kFullMask, m, off));
        double sum = 0.0;
        for (int e = lane; e < E; e += 32) {
            const double v = exp(pv[e] - m);
            pv[e] = v;
            sum += v;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFullMask, sum, off);
        for (int e = lane; e < E; e += 32) pv[e] /= sum;
    } else {
        for (int e = lane; e < E; e += 32) pv[e] = 1.0 / (1.0 + exp(-pv[e]));
    }
    __syncwarp();
    uint32_t kmask = kFullMask;
    int G = E;
    if (a.n_group > 1) {
        const int ng = a.n_group;
        G = E / ng;
        double gs = -DBL_MAX;
        if (lane < ng) {
            double s1 = -DBL_MAX, s2 = -DBL_MAX;
            for (int e = lane * G; e < (lane + 1) * G; ++e) {
                const double v = pv[e] + static_cast<double>(a.bias[e]);
                if (v > s1) { s2 = s1; s1 = v; } else if (v > s2) { s2 = v; }
            }
            gs = a.group_top == 2 ? s1 + s2 : s1;
        }
        kmask = 0u;
        bool in = lane < ng;
        for (int r = 0; r < a.topk_group; ++r) {
            double bs = in ? gs : -DBL_MAX;
            int bg = in ? lane : INT_MAX;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const double os = __shfl_xor_sync(kFullMask, bs, off);
                const int og = __shfl_xor_sync(kFullMask, bg, off);
                if (og != INT_MAX && (bg == INT_MAX || before64(os, og, bs, bg))) { bs = os; bg = og; }
            }
            if (bg == INT_MAX) break;          // (topk_group <= n_group: not reached)
            kmask |= 1u << bg;
            if (lane == bg) in = false;
        }
    }
    for (int j = 0; j < K; ++j) {
        double bs = -DBL_MAX;
        int be = INT_MAX;
        for (int e = lane; e < E; e += 32) {
            if (pe[e] < 0 || !((kmask >> (e / G)) & 1u)) continue;
            const double v = pv[e] + static_cast<double>(a.bias[e]);
            if (be == INT_MAX || before64(v, e, bs, be)) { bs = v; be = e; }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const double os = __shfl_xor_sync(kFullMask, bs, off);
            const int oe = __shfl_xor_sync(kFullMask, be, off);
            if (oe != INT_MAX && (be == INT_MAX || before64(os, oe, bs, be))) { bs = os; be = oe; }
        }
        if (be == INT_MAX) be = 0;        // (no candidate left: cannot happen for K <= E)
        if (lane == 0) ord[j] = be;
        __syncwarp();
        if (lane == (be & 31)) pe[be] = -1 - be;
        __syncwarp();
    }
    double den = 0.0;
    for (int j = 0; j < K; ++j) den += pv[ord[j]];
    for (int j = lane; j < K; j += 32) {
        const int e = ord[j];
        oi[j] = e;
        ow[j] = static_cast<float>(a.renorm ? pv[e] / den : pv[e]);
    }
    __syncwarp();
}

// Candidate bits of every expert (the general options re-score all of them).
__device__ __forceinline__ uint32_t all_experts(int E, int lane)
{
    const int NI = (E + 31) / 32;
    uint32_t c = 0;
    for (int i = 0; i < NI; ++i)
        if (lane + 32 * i < E) c |= 1u << i;
    return c;
}

// Writes the lane-distributed candidate bits of a token as a compact expert list.
__device__ int list_candidates(uint32_t cand, int E, int *out, int lane)
{
    const int NI = (E + 31) / 32;
    int pos = 0;
    for (int i = 0; i < NI; ++i) {
        const bool c = (cand >> i) & 1u;
        const uint32_t m = __ballot_sync(kFullMask, c);
        if (c) out[pos + __popc(m & ((1u << lane) - 1u))] = lane + 32 * i;
        pos += __popc(m);
    }
    __syncwarp();
    return pos;
}

// ------------------------------------------------------------------------ tile GEMM
// Computes the fp32 logit tile of CTA (et, tt, ks) and the squared norms of its slices.
template <class C>
__device__ void gemm_tile(const RouterArgs &a, unsigned char *smem)
{
    const int et = blockIdx.x, tt = blockIdx.y, ks = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = tt * C::TT, e0 = et * C::TE;
    const int s_beg = static_cast<int>(static_cast<long long>(ks) * a.S / a.KS);
    const int s_end = static_cast<int>(static_cast<long long>(ks + 1) * a.S / a.KS);

    float *xs = reinterpret_cast<float *>(smem);   // [2][KST][TT]
    float *wsm = xs + 2 * KST * C::TT;             // [2][KST][TE]

    // loaders: vector q -> (row q % ROWS, 8-element group q / ROWS); consecutive threads
    // take consecutive rows, so the transposed shared-memory stores do not conflict
    const uint4 *xp[C::XPT];
    bool xok[C::XPT];
#pragma unroll
    for (int i = 0; i < C::XPT; ++i) {
        const int q = tid + NT * i;
        const int row = t0 + q % C::TT;
        xok[i] = q < C::XV && row < a.T;
        xp[i] = reinterpret_cast<const uint4 *>(a.X + static_cast<size_t>(xok[i] ? row : 0) * a.H) + q / C::TT;
    }
    const uint4 *wp[C::WPT];
    bool wok[C::WPT];
#pragma unroll
    for (int i = 0; i < C::WPT; ++i) {
        const int q = tid + NT * i;
        const int row = e0 + q % C::TE;
        wok[i] = q < C::WV && row < a.E;
        wp[i] = reinterpret_cast<const uint4 *>(a.Wg + static_cast<size_t>(wok[i] ? row : 0) * a.H) + q / C::TE;
    }
    float xsq[C::XPT], wsq[C::WPT];
#pragma unroll
    for (int i = 0; i < C::XPT; ++i) xsq[i] = 0.f;
#pragma unroll
    for (int i = 0; i < C::WPT; ++i) wsq[i] = 0.f;

    uint4 rx[C::PF][C::XPT], rw[C::PF][C::WPT];    // register ring of prefetched stages
    auto gload = [&](int j, int st) {
#pragma unroll
        for (int i = 0; i < C::XPT; ++i) rx[j][i] = xok[i] ? __ldg(xp[i] + st * 4) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < C::WPT; ++i) rw[j][i] = wok[i] ? __ldg(wp[i] + st * 4) : make_uint4(0, 0, 0, 0);
    };
    auto sstore = [&](int j, int buf) {
#pragma unroll
        for (int i = 0; i < C::XPT; ++i) {
            const int q = tid + NT * i;
            if (q < C::XV) {
                float f[8];
                unpack8(rx[j][i], f);
                float *d = xs + buf * KST * C::TT + ((q / C::TT) * 8) * C::TT + q % C::TT;
#pragma unroll
                for (int e = 0; e < 8; ++e) { d[e * C::TT] = f[e]; xsq[i] = fmaf(f[e], f[e], xsq[i]); }
            }
        }
#pragma unroll
        for (int i = 0; i < C::WPT; ++i) {
            const int q = tid + NT * i;
            if (q < C::WV) {
                float f[8];
                unpack8(rw[j][i], f);
                float *d = wsm + buf * KST * C::TE + ((q / C::TE) * 8) * C::TE + q % C::TE;
#pragma unroll
                for (int e = 0; e < 8; ++e) { d[e * C::TE] = f[e]; wsq[i] = fmaf(f[e], f[e], wsq[i]); }
            }
        }
    };

    // output micro-tile of this thread: TPT tokens and EPT experts, each in groups of four
    // interleaved over the warp's lane rows (LY) and lane columns (LX): token group g of
    // lane row r is wtok + 4 (LY g + r) ..+3, expert group g of lane column c is
    // wexp + 4 (LX g + c) ..+3, so each 16-byte operand read covers one contiguous span of
    // the stage across the warp
    constexpr int WY = C::NTY / C::LY;
    constexpr int LX = 32 / C::LY;
    const int wtok = (warp % WY) * (C::LY * C::TPT) + 4 * (lane % C::LY);
    const int wexp = (warp / WY) * (LX * C::EPT) + 4 * (lane / C::LY);
    auto tok = [&](int i) { return wtok + (i >> 2) * (4 * C::LY) + (i & 3); };
    auto exq = [&](int j) { return wexp + (j >> 2) * (4 * LX) + (j & 3); };
    float acc[C::TPT * C::EPT];
#pragma unroll
    for (int p = 0; p < C::TPT * C::EPT; ++p) acc[p] = 0.f;

#pragma unroll
    for (int j = 0; j < C::PF; ++j)
        if (s_beg + j < s_end) gload(j, s_beg + j);
    for (int s0 = s_beg; s0 < s_end; s0 += C::PF) {
#pragma unroll
        for (int j = 0; j < C::PF; ++j) {
            const int st = s0 + j;
            if (st < s_end) {
                const int buf = st & 1;
                sstore(j, buf);
                if (st + C::PF < s_end) gload(j, st + C::PF);
                __syncthreads();
                // one 32-deep fp32 chain per (token, expert) for this stage, then added to
                // the running sum of the split
                const float *xb = xs + buf * KST * C::TT + wtok;
                const float *wb = wsm + buf * KST * C::TE + wexp;
                float acc_in[C::TPT * C::EPT];
#pragma unroll
                for (int q = 0; q < C::TPT * C::EPT; ++q) acc_in[q] = 0.f;
#pragma unroll 4
                for (int kk = 0; kk < KST; ++kk) {
                    float xa[C::TPT];
#pragma unroll
                    for (int i4 = 0; i4 < C::TPT / 4; ++i4) {
                        const float4 v = *reinterpret_cast<const float4 *>(xb + kk * C::TT + 4 * C::LY * i4);
                        xa[4 * i4] = v.x; xa[4 * i4 + 1] = v.y; xa[4 * i4 + 2] = v.z; xa[4 * i4 + 3] = v.w;
                    }
                    const float4 wv = *reinterpret_cast<const float4 *>(wb + kk * C::TE);
                    const float wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int i = 0; i < C::TPT; ++i)
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            acc_in[i * 4 + jj] = fmaf(xa[i], wa[jj], acc_in[i * 4 + jj]);
                }
#pragma unroll
                for (int q = 0; q < C::TPT * C::EPT; ++q) acc[q] += acc_in[q];
            }
        }
    }

#pragma unroll
    for (int i = 0; i < C::TPT; ++i) {
        const int t = t0 + tok(i);
        if (t >= a.T) continue;
        float *dst = a.part + (static_cast<size_t>(ks) * a.T + t) * a.E;
#pragma unroll
        for (int g = 0; g < C::EPT / 4; ++g) {
            const int e = e0 + exq(4 * g);
            const float *v = acc + i * C::EPT + 4 * g;
            if ((a.E & 3) == 0 && e + 3 < a.E) {
                *reinterpret_cast<float4 *>(dst + e) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    if (e + jj < a.E) dst[e + jj] = v[jj];
            }
        }
    }

    // squared norms of this slice, reduced over the four 8-element groups of a row in order
    __syncthreads();
    float *rxs = xs;                   // [4][TT]
    float *rws = xs + 4 * C::TT;       // [4][TE]
#pragma unroll
    for (int i = 0; i < C::XPT; ++i) {
        const int q = tid + NT * i;
        if (q < C::XV) rxs[q] = xsq[i];
    }
#pragma unroll
    for (int i = 0; i < C::WPT; ++i) {
        const int q = tid + NT * i;
        if (q < C::WV) rws[q] = wsq[i];
    }
    __syncthreads();
    for (int r = tid; r < C::TT; r += NT) {
        const float sx = ((rxs[r] + rxs[C::TT + r]) + rxs[2 * C::TT + r]) + rxs[3 * C::TT + r];
        if (et == 0 && t0 + r < a.T) a.xsq[static_cast<size_t>(ks) * a.T + t0 + r] = sx;
    }
    for (int r = tid; r < C::TE; r += NT) {
        const float sw = ((rws[r] + rws[C::TE + r]) + rws[2 * C::TE + r]) + rws[3 * C::TE + r];
        if (e0 + r < a.E) a.wsq[(static_cast<size_t>(tt) * a.KS + ks) * a.E + e0 + r] = sw;
    }
}

// ------------------------------------------------- warp-specialised tile GEMM (large)
// The large-batch tile with its operand traffic taken off the compute warps: four producer
// warps load the bf16 token and gate-row slices of each stage, convert them to fp32 into
// a ring of WS stages (the same transposed layout) and keep the slices' squared norms; the
// eight compute warps only run the 32-deep chains (the same operations in the same order
// as gemm_tile, so the logits and the bound are unchanged).  full[s] / empty[s] mbarriers
// hand the stages over; every wait is bounded and, on expiry, records
// MOE_ERR_DEVICE_TIMEOUT and makes both roles leave their loops.
constexpr int NPW = 4;             // producer warps (one per SM sub-partition)
constexpr int NT_WS = NT + 32 * NPW;   // eight compute warps + the producer warps
constexpr unsigned long long kWsWaitNs = 1000000000ull;

template <class C>
__host__ __device__ constexpr size_t ws_smem_bytes()
{
    constexpr int PT = 32 * NPW;
    constexpr int XI = 4 * ((C::TT + PT - 1) / PT), WI = 4 * ((C::TE + PT - 1) / PT);
    constexpr int XP = C::TT < PT ? C::TT : PT;       // producer threads with token units
    return static_cast<size_t>(C::RING) * KST * (C::TT + C::TE) * sizeof(float) +
           static_cast<size_t>(C::STG) * (XI * XP + WI * PT) * 16 + 2 * C::RING * 8 + 16;
}

// 16-byte global -> shared copy, zero-filled when !valid (src must still be addressable).
__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 16 : 0) : "memory");
}

template <class C>
__device__ void gemm_tile_ws(const RouterArgs &a, unsigned char *smem)
{
    constexpr int PT = 32 * NPW;                                // producer threads
    constexpr int WS = C::RING, WSB = C::STG;
    // producer units: 4 consecutive rows x one 8-element group of a stage (TT units for
    // the token slice, TE for the gate rows; a tile smaller than PT leaves threads idle)
    static_assert((C::TT % PT == 0 || C::TT < PT) && C::TE % PT == 0, "warp-specialised tile");
    constexpr int XU = (C::TT + PT - 1) / PT, WU = C::TE / PT;  // units a producer thread
    constexpr int XI = 4 * XU, WI = 4 * WU;                     // 16-byte vectors a thread
    constexpr int XP = C::TT < PT ? C::TT : PT;                 // threads with token units
    constexpr int SV = XI * XP + WI * PT;                       // staged vectors a stage
    const int et = blockIdx.x, tt = blockIdx.y, ks = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = tt * C::TT, e0 = et * C::TE;
    const int s_beg = static_cast<int>(static_cast<long long>(ks) * a.S / a.KS);
    const int s_end = static_cast<int>(static_cast<long long>(ks + 1) * a.S / a.KS);
    const int n_st = s_end - s_beg;

    float *xs = reinterpret_cast<float *>(smem);                  // [WS][KST][TT]
    float *wsm = xs + WS * KST * C::TT;                           // [WS][KST][TE]
    // staging ring: per stage [XI][XP] token vectors, then [WI][PT] gate-row vectors
    uint4 *stg = reinterpret_cast<uint4 *>(wsm + WS * KST * C::TE);
    uint64_t *full = reinterpret_cast<uint64_t *>(stg + WSB * SV);
    uint64_t *empty = full + WS;
    int *abort_flag = reinterpret_cast<int *>(empty + WS);
    if (tid == 0) {
        for (int s = 0; s < WS; ++s) {
            mbar_init(&full[s], PT);
            mbar_init(&empty[s], NW);
        }
        *abort_flag = 0;
    }
    __syncthreads();
    volatile int *abort_v = abort_flag;

    float xsq[XI], wsq[WI];        // producer: squared norms of (row, group) slices
    constexpr int WY = C::NTY / C::LY;
    constexpr int LX = 32 / C::LY;
    const int wtok = (warp % WY) * (C::LY * C::TPT) + 4 * (lane % C::LY);
    const int wexp = (warp / WY) * (LX * C::EPT) + 4 * (lane / C::LY);
    auto tok = [&](int i) { return wtok + (i >> 2) * (4 * C::LY) + (i & 3); };
    auto exq = [&](int j) { return wexp + (j >> 2) * (4 * LX) + (j & 3); };
    uint64_t accp[C::TPT / 2 * C::EPT];

    const int ptid = tid - NT;   // producer thread index (>= 0 in the producer warps)
    if (warp >= NW) {
        // ----------------------------------------------------------- producer warps
        // unit u = ptid + PT i: rows 4 (u % (TT / 4)) ..+3, 8-element group u / (TT / 4);
        // consecutive threads take consecutive row quads, so the 16-byte transposed stores
        // (four rows at one k) of a warp cover one contiguous span
#pragma unroll
        for (int i = 0; i < XI; ++i) xsq[i] = 0.f;
#pragma unroll
        for (int i = 0; i < WI; ++i) wsq[i] = 0.f;
        // raw bf16 slices land in a staging ring by cp.async, WSB - 1 stages ahead; each
        // thread converts the 16-byte vectors it copied itself
        auto copy_stage = [&](int n) {
            if (n < n_st) {
                const int st = s_beg + n;
                uint4 *sb = stg + (n % WSB) * SV;
#pragma unroll
                for (int i = 0; i < XU; ++i) {
                    const int u = ptid + PT * i, r0 = 4 * (u % (C::TT / 4)), g = u / (C::TT / 4);
                    if (u >= C::TT) break;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int row = t0 + r0 + q;
                        const uint4 *src = reinterpret_cast<const uint4 *>(a.X + static_cast<size_t>(row < a.T ? row : 0) * a.H) + st * 4 + g;
                        cp_async16(sb + (4 * i + q) * XP + ptid, src, row < a.T);
                    }
                }
#pragma unroll
                for (int i = 0; i < WU; ++i) {
                    const int u = ptid + PT * i, r0 = 4 * (u % (C::TE / 4)), g = u / (C::TE / 4);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int row = e0 + r0 + q;
                        const uint4 *src = reinterpret_cast<const uint4 *>(a.Wg + static_cast<size_t>(row < a.E ? row : 0) * a.H) + st * 4 + g;
                        cp_async16(sb + XI * XP + (4 * i + q) * PT + ptid, src, row < a.E);
                    }
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        // four rows of one group -> eight 16-byte stores (one per k) and the rows' norms
        auto convert = [&](const uint4 *sv, int sstride, float *dst, int ld, float *nrm) {
            float f[4][8];
#pragma unroll
            for (int q = 0; q < 4; ++q) unpack8(sv[q * sstride], f[q]);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                *reinterpret_cast<float4 *>(dst + k * ld) = make_float4(f[0][k], f[1][k], f[2][k], f[3][k]);
#pragma unroll
                for (int q = 0; q < 4; ++q) nrm[q] = fmaf(f[q][k], f[q][k], nrm[q]);
            }
        };
#pragma unroll
        for (int n = 0; n < WSB - 1; ++n) copy_stage(n);
        for (int n = 0; n < n_st; ++n) {
            const int slot = n % WS;
            copy_stage(n + WSB - 1);
            asm volatile("cp.async.wait_group %0;" ::"n"(WSB - 1) : "memory");
            // (warp-uniform: a lane that gave up takes the whole warp out of the loop)
            if (n >= WS && !__all_sync(kFullMask, mbar_wait(&empty[slot], ((n / WS) - 1) & 1, abort_v,
                                                             a.status, kWsWaitNs)))
                break;
            const uint4 *sb = stg + (n % WSB) * SV + ptid;
            float *xd = xs + slot * KST * C::TT;
            float *wd = wsm + slot * KST * C::TE;
#pragma unroll
            for (int i = 0; i < XU; ++i) {
                const int u = ptid + PT * i, r0 = 4 * (u % (C::TT / 4)), g = u / (C::TT / 4);
                if (u < C::TT) convert(sb + 4 * i * XP, XP, xd + g * 8 * C::TT + r0, C::TT, xsq + 4 * i);
            }
#pragma unroll
            for (int i = 0; i < WU; ++i) {
                const int u = ptid + PT * i, r0 = 4 * (u % (C::TE / 4)), g = u / (C::TE / 4);
                convert(sb + XI * XP + 4 * i * PT, PT, wd + g * 8 * C::TE + r0, C::TE, wsq + 4 * i);
            }
            mbar_arrive(&full[slot]);
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    } else {
        // ------------------------------------------------------------ compute warps
#pragma unroll
        for (int q = 0; q < C::TPT / 2 * C::EPT; ++q) accp[q] = 0ull;
        for (int n = 0; n < n_st; ++n) {
            const int slot = n % WS;
            if (!__all_sync(kFullMask, mbar_wait(&full[slot], (n / WS) & 1, abort_v, a.status, kWsWaitNs)))
                break;
            const float *xb = xs + slot * KST * C::TT + wtok;
            const float *wb = wsm + slot * KST * C::TE + wexp;
            // pair pp * EPT + jj = (token 2pp, token 2pp + 1) x expert jj
            uint64_t pin[C::TPT / 2 * C::EPT];
#pragma unroll
            for (int q = 0; q < C::TPT / 2 * C::EPT; ++q) pin[q] = 0ull;
#pragma unroll 4
            for (int kk = 0; kk < KST; ++kk) {
                ulonglong2 xv[C::TPT / 4];
#pragma unroll
                for (int i4 = 0; i4 < C::TPT / 4; ++i4)
                    xv[i4] = *reinterpret_cast<const ulonglong2 *>(xb + kk * C::TT + 4 * C::LY * i4);
                uint64_t wp[C::EPT];
#pragma unroll
                for (int g = 0; g < C::EPT / 4; ++g) {
                    const float4 wv = *reinterpret_cast<const float4 *>(wb + kk * C::TE + 4 * LX * g);
                    wp[4 * g] = dup_x2(wv.x);
                    wp[4 * g + 1] = dup_x2(wv.y);
                    wp[4 * g + 2] = dup_x2(wv.z);
                    wp[4 * g + 3] = dup_x2(wv.w);
                }
#pragma unroll
                for (int pp = 0; pp < C::TPT / 2; ++pp) {
                    const uint64_t xp = (pp & 1) ? xv[pp >> 1].y : xv[pp >> 1].x;
#pragma unroll
                    for (int jj = 0; jj < C::EPT; ++jj)
                        pin[pp * C::EPT + jj] = fma_x2(xp, wp[jj], pin[pp * C::EPT + jj]);
                }
            }
#pragma unroll
            for (int q = 0; q < C::TPT / 2 * C::EPT; ++q) accp[q] = add_x2(accp[q], pin[q]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }
    __syncthreads();

    if (warp < NW) {
        float *part_t = a.part + static_cast<size_t>(ks) * a.T * a.E;
#pragma unroll
        for (int pp = 0; pp < C::TPT / 2; ++pp) {
            const int tA = t0 + tok(2 * pp), tB = t0 + tok(2 * pp + 1);
#pragma unroll
            for (int g = 0; g < C::EPT / 4; ++g) {
                const int e = e0 + exq(4 * g);
                float lo[4], hi[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo[jj]), "=f"(hi[jj]) : "l"(accp[pp * C::EPT + 4 * g + jj]));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = h ? tB : tA;
                    const float *v = h ? hi : lo;
                    if (t >= a.T) continue;
                    float *dst = part_t + static_cast<size_t>(t) * a.E;
                    if ((a.E & 3) == 0 && e + 3 < a.E) {
                        *reinterpret_cast<float4 *>(dst + e) = make_float4(v[0], v[1], v[2], v[3]);
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            if (e + jj < a.E) dst[e + jj] = v[jj];
                    }
                }
            }
        }
    } else {
        // squared norms of this slice, reduced over the four 8-element groups of a row
        float *rxs = xs;                   // [4][TT]
        float *rws = xs + 4 * C::TT;       // [4][TE]
#pragma unroll
        for (int i = 0; i < XU; ++i) {
            const int u = ptid + PT * i, r0 = 4 * (u % (C::TT / 4)), g = u / (C::TT / 4);
            if (u >= C::TT) break;
#pragma unroll
            for (int q = 0; q < 4; ++q) rxs[g * C::TT + r0 + q] = xsq[4 * i + q];
        }
#pragma unroll
        for (int i = 0; i < WU; ++i) {
            const int u = ptid + PT * i, r0 = 4 * (u % (C::TE / 4)), g = u / (C::TE / 4);
#pragma unroll
            for (int q = 0; q < 4; ++q) rws[g * C::TE + r0 + q] = wsq[4 * i + q];
        }
        asm volatile("bar.sync 1, %0;" ::"n"(PT) : "memory");   // the producer warps only
        for (int r = ptid; r < C::TT; r += PT) {
            const float sx = ((rxs[r] + rxs[C::TT + r]) + rxs[2 * C::TT + r]) + rxs[3 * C::TT + r];
            if (et == 0 && t0 + r < a.T) a.xsq[static_cast<size_t>(ks) * a.T + t0 + r] = sx;
        }
        for (int r = ptid; r < C::TE; r += PT) {
            const float sw = ((rws[r] + rws[C::TE + r]) + rws[2 * C::TE + r]) + rws[3 * C::TE + r];
            if (e0 + r < a.E) a.wsq[(static_cast<size_t>(tt) * a.KS + ks) * a.E + e0 + r] = sw;
        }
    }
}

// ----------------------------------------------------------- tiny batches (T <= 8)
// GEMV_QW warps share one expert's gate row, each reading a quarter of it once and forming
// the partial logits of all T tokens; a CTA holds GEMV_EPC experts, so the whole gate
// matrix is read by E * GEMV_QW warps spread over the GPU (a cold read of 3.7 MB is
// latency-bound: it needs many loads in flight).  Each partial is 8 independent fp32
// chains (one per element of a 16-byte vector) added by a fixed 3-level tree and a
// 5-level warp tree; the quarters are added by a fixed 2-level tree.
constexpr int GEMV_TMAX = 8;      // up to 8 tokens (5..8: 87 -> 65 us per router stage than the
                                  // 16x256 tile path, which has one CTA per split here)
constexpr int GEMV_QW = 4;        // warps per gate row
constexpr int GEMV_EPC = NW / GEMV_QW;

template <int TB>     // token batch: 1, 2, 4 or 8 (>= T)
__device__ void gemv_tile(const RouterArgs &a, unsigned char *smem)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int el = warp / GEMV_QW, qw = warp % GEMV_QW;
    const int e = blockIdx.x * GEMV_EPC + el;
    const int T = a.T, nv = a.H / 8;
    const int v_beg = nv * qw / GEMV_QW, v_end = nv * (qw + 1) / GEMV_QW;
    constexpr int RS = 2 * TB + 1;                    // per warp: dots, gate norm, token norms
    float *red = reinterpret_cast<float *>(smem);     // [NW][RS]
    if (e < a.E) {
        const uint4 *wr = reinterpret_cast<const uint4 *>(a.Wg + static_cast<size_t>(e) * a.H);
        const uint4 *xr = reinterpret_cast<const uint4 *>(a.X);
        float acc[TB][8], xq[TB];
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            xq[t] = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[t][j] = 0.f;
        }
        float wsq = 0.f;
        // vectors per lane in flight: a quarter row of DeepSeek-V3's gate (224 vectors) in
        // one round trip for one or two tokens
        constexpr int U = TB <= 2 ? 8 : (TB <= 4 ? 4 : 2);
        for (int v0 = v_beg + lane; v0 < v_end; v0 += 32 * U) {
            uint4 wv[U], xv[U][TB];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + 32 * u;
                const bool ok = v < v_end;
                wv[u] = ok ? __ldg(wr + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int t = 0; t < TB; ++t)
                    xv[u][t] = (ok && t < T) ? __ldg(xr + static_cast<size_t>(t) * nv + v)
                                             : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float wf[8];
                unpack8(wv[u], wf);
#pragma unroll
                for (int j = 0; j < 8; ++j) wsq = fmaf(wf[j], wf[j], wsq);
#pragma unroll
                for (int t = 0; t < TB; ++t) {
                    float xf[8];
                    unpack8(xv[u][t], xf);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        acc[t][j] = fmaf(xf[j], wf[j], acc[t][j]);
                        xq[t] = fmaf(xf[j], xf[j], xq[t]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            float sum = ((acc[t][0] + acc[t][1]) + (acc[t][2] + acc[t][3])) +
                        ((acc[t][4] + acc[t][5]) + (acc[t][6] + acc[t][7]));
            float q = xq[t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                sum += __shfl_xor_sync(kFullMask, sum, off);
                q += __shfl_xor_sync(kFullMask, q, off);
            }
            if (lane == 0) {
                red[warp * RS + t] = sum;
                red[warp * RS + TB + 1 + t] = q;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) wsq += __shfl_xor_sync(kFullMask, wsq, off);
        if (lane == 0) red[warp * RS + TB] = wsq;
    }
    __syncthreads();
    // quarters -> logits, gate norms and (once, in CTA 0) token norms
    auto quarters = [&](int elx, int k) {
        const float *r = red + elx * GEMV_QW * RS + k;
        return (r[0] + r[RS]) + (r[2 * RS] + r[3 * RS]);
    };
    static_assert(GEMV_QW == 4, "the quarter tree adds four partials");
    const int tid = threadIdx.x;
    if (tid < GEMV_EPC * TB) {
        const int elx = tid / TB, t = tid % TB, ex = blockIdx.x * GEMV_EPC + elx;
        if (ex < a.E && t < T) a.part[static_cast<size_t>(t) * a.E + ex] = quarters(elx, t);
    } else if (tid < GEMV_EPC * TB + GEMV_EPC) {
        const int elx = tid - GEMV_EPC * TB, ex = blockIdx.x * GEMV_EPC + elx;
        if (ex < a.E) a.wsq[ex] = quarters(elx, TB);
    } else if (blockIdx.x == 0 && tid < GEMV_EPC * TB + GEMV_EPC + TB) {
        const int t = tid - GEMV_EPC * TB - GEMV_EPC;
        if (t < T) a.xsq[t] = quarters(0, TB + 1 + t);
    }
}

// Re-scores the listed (token, expert) pairs of a CTA -- p_tok[q] >= 0 a token relative to
// t0, p_e[q] >= 0 an expert; other entries are skipped -- in double-word arithmetic with all
// of the CTA's warps, and writes p_val[q]: the fp64 logit (routing options) or sigmoid +
// bias.  With fewer pairs than warps, each dot product is split over a group of 2, 4 or 8
// warps (ranges of H, partials merged in rank order), so a re-score costs about one memory
// round trip.  CTA-wide: every thread calls it.  Scratch: need [npairs] ints, dwp [NW],
// s_n one shared int.
__device__ void rescore_pairs(const RouterArgs &a, const int *p_e, const int *p_tok, int npairs,
                              int t0, const float *bias, int *need, float2 *dwp, double *p_val,
                              int *s_n, int warp, int lane)
{
    if (warp == 0) {
        int n = 0;
        for (int q0 = 0; q0 < npairs; q0 += 32) {
            const int q = q0 + lane;
            const bool nd = q < npairs && p_e[q] >= 0 && p_tok[q] >= 0;
            const uint32_t m = __ballot_sync(kFullMask, nd);
            if (nd) need[n + __popc(m & ((1u << lane) - 1u))] = q;
            n += __popc(m);
        }
        if (lane == 0) *s_n = n;
    }
    __syncthreads();
    const int nneed = *s_n;
    if (nneed == 0) return;
    // group size: 8 warps on one pair, 4 on each of two, 2 on each of four, else one
    const int G = nneed >= NW ? 1 : (nneed >= NW / 2 ? 2 : (nneed >= 2 ? 4 : 8));
    const int rank = warp % G, slot = warp / G, per_round = NW / G;
    const int nv = a.H / 8;
    const int v0 = rank * nv / G, v1 = (rank + 1) * nv / G;
    for (int r0 = 0; r0 < nneed; r0 += per_round) {
        const int i = r0 + slot;
        if (i < nneed) {
            const int q = need[i];
            const int e = p_e[q], t = t0 + p_tok[q];
            float h, l;
            dot_dw_range(a.X + static_cast<size_t>(t) * a.H, a.Wg + static_cast<size_t>(e) * a.H,
                         v0, v1, lane, h, l);
            if (lane == 0) dwp[warp] = make_float2(h, l);
        }
        __syncthreads();
        if (i < nneed && rank == 0 && lane == 0) {
            float h = dwp[warp].x, l = dwp[warp].y;
            for (int g = 1; g < G; ++g) dw_merge(h, l, dwp[warp + g].x, dwp[warp + g].y);
            const double l64 = static_cast<double>(h) + static_cast<double>(l);
            const int q = need[i];
            p_val[q] = a.variant ? l64 : 1.0 / (1.0 + exp(-l64)) + static_cast<double>(bias[p_e[q]]);
        }
        __syncthreads();
    }
}

// Shared-memory layout of the finalise step (after the GEMM tile is done with smem).
struct FinSmem {
    float *nw, *bias, *nxs, *L;        // [E], [E], [CH], [CH][E]
    float *sel, *bnd, *sc;             // per warp [E] each
    int *ord, *ce;                     // per warp [32], [E]
    int *p_e, *p_tok, *need;           // refine list [max_pairs] x 3
    double *p_val, *s64;               // [max_pairs], per warp [E]
    float2 *dwp;                       // [NW] partial double-word dots

    __device__ FinSmem(unsigned char *smem, int E, int max_pairs, int warp)
    {
        float *f = reinterpret_cast<float *>(smem);
        dwp = reinterpret_cast<float2 *>(f); f += 2 * NW;   // (first: 8-byte aligned)
        nw = f; f += E;
        bias = f; f += E;
        nxs = f; f += CH;
        L = f; f += CH * E;
        sel = f + static_cast<size_t>(warp) * 3 * E;
        bnd = sel + E;
        sc = bnd + E;
        f += NW * 3 * E;
        int *i = reinterpret_cast<int *>(f);
        ord = i + warp * 32; i += NW * 32;
        ce = i + static_cast<size_t>(warp) * E; i += NW * E;
        p_e = i; i += max_pairs;
        p_tok = i; i += max_pairs;
        need = i; i += max_pairs;
        const uintptr_t d = (reinterpret_cast<uintptr_t>(i) + 7) & ~static_cast<uintptr_t>(7);
        p_val = reinterpret_cast<double *>(d);
        s64 = p_val + max_pairs + static_cast<size_t>(warp) * E;
    }
    static size_t bytes(int E, int max_pairs)
    {
        return (2 * NW + 2 * static_cast<size_t>(E) + CH + static_cast<size_t>(CH) * E +
                static_cast<size_t>(NW) * 3 * E) * 4 +
               (NW * 32 + static_cast<size_t>(NW) * E + 3 * static_cast<size_t>(max_pairs)) * 4 + 8 +
               (static_cast<size_t>(max_pairs) + static_cast<size_t>(NW) * E) * 8;
    }
};

// Refines one token with its warp alone (used when the shared list is full, and by the
// one-warp-per-token finaliser).
__device__ void refine_token_warp(const RouterArgs &a, int t, uint32_t cand, int *ce,
                                  double *s64, int *ord, int lane, bool every = false,
                                  uint32_t ck = kFullMask, uint32_t ug = 0u)
{
    const int nc = list_candidates(cand, a.E, ce, lane);
    const uint16_t *xrow = a.X + static_cast<size_t>(t) * a.H;
    for (int q = 0; q < nc; ++q) {
        const int e = ce[q];
        const double l64 = dot_double_word(xrow, a.Wg + static_cast<size_t>(e) * a.H, a.H, lane);
        if (lane == 0)
            s64[q] = a.variant ? l64 : 1.0 / (1.0 + exp(-l64)) + static_cast<double>(a.bias[e]);
    }
    __syncwarp();
    if (a.variant && every)
        select_general64(a, ce, s64, a.topk_idx + static_cast<size_t>(t) * a.K,
                         a.topk_w + static_cast<size_t>(t) * a.K, ord, lane);
    else if (a.variant)
        select_candidates64(a, ce, s64, nc, ck, ug, a.topk_idx + static_cast<size_t>(t) * a.K,
                            a.topk_w + static_cast<size_t>(t) * a.K, ord, lane);
    else
        select_refined(ce, s64, nc, a.K, a.bias, a.topk_idx + static_cast<size_t>(t) * a.K,
                       a.topk_w + static_cast<size_t>(t) * a.K, ord, lane);
}

// Whether the lane's candidate (of at most 32) has an interval [sel - bound, sel + bound]
// that meets another candidate's.  Only those need re-scoring: a candidate whose interval
// is disjoint from all the others keeps its fp32 sel, which lies in that interval, so it
// orders against any candidate exactly as the exact value would.  Default routing options.
__device__ bool meets_another(const int *ce, int nc, const float *w_sel, const float *w_bnd, int lane)
{
    const int e = lane < nc ? ce[lane] : 0;
    const float lo = lane < nc ? __fsub_rd(w_sel[e], w_bnd[e]) : FLT_MAX;
    const float hi = lane < nc ? __fadd_ru(w_sel[e], w_bnd[e]) : -FLT_MAX;
    bool meets = false;
    for (int r = 0; r < nc; ++r) {
        const float olo = __shfl_sync(kFullMask, lo, r), ohi = __shfl_sync(kFullMask, hi, r);
        meets |= r != lane && lo <= ohi && olo <= hi;
    }
    return meets;
}

// ------------------------------------------------------- fused kernel (small batches)
template <class C, int GEMV>   // GEMV = token batch of the tiny-batch path, 0 = tile GEMM
__global__ void __launch_bounds__(NT, 2) router_fused_kernel(const RouterArgs a)
{
    pdl_wait();
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_last, s_npairs, s_npend, s_nneed;
    __shared__ int s_pend[5 * C::TT];     // (token, first pair, pair count, ck, ug) to refine

    if constexpr (GEMV > 0)
        gemv_tile<GEMV>(a, smem);
    else
        gemm_tile<C>(a, smem);

    // ---------------------------------------------------------- last CTA finalises
    const int tt = blockIdx.y, tid = threadIdx.x;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&a.cnt[tt], 1u);
        s_last = (prev == static_cast<unsigned>(gridDim.x * gridDim.z - 1));
        s_npairs = 0;
        s_npend = 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    const int warp = tid >> 5, lane = tid & 31;
    const int E = a.E, KS = a.KS, t0 = tt * C::TT;
    FinSmem S(smem, E, a.max_pairs, warp);
    const Bounds bd(a.depth, KS, a.H);
    for (int e = tid; e < E; e += NT) {        // gate-row norms and biases, once per CTA
        float nw2 = 0.f;
        for (int q0 = 0; q0 < KS; q0 += 16) {  // splits in batches of 16 loads, added in order
            float w[16];
#pragma unroll
            for (int q = 0; q < 16; ++q)
                if (q0 + q < KS) w[q] = __ldcg(a.wsq + (static_cast<size_t>(tt) * KS + q0 + q) * E + e);
#pragma unroll
            for (int q = 0; q < 16; ++q)
                if (q0 + q < KS) nw2 += w[q];
        }
        S.nw[e] = sqrtf(nw2) * bd.infl;
        S.bias[e] = a.bias[e];
    }

    for (int c0 = 0; c0 < C::TT; c0 += CH) {
        __syncthreads();
        // K-split partials of the chunk's tokens -> shared logits (fixed order over splits)
        const int n4 = (E & 3) == 0 ? E / 4 : 0;
        if (n4) {
            // up to 16 independent loads in flight per thread, added in split order
            const size_t stride = static_cast<size_t>(a.T) * E / 4;
            for (int it = tid; it < CH * n4; it += NT) {
                const int tl = it / n4, g = it - tl * n4, t = t0 + c0 + tl;
                if (t >= a.T) continue;
                const float4 *src = reinterpret_cast<const float4 *>(a.part + static_cast<size_t>(t) * E) + g;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int q0 = 0; q0 < KS; q0 += 16) {   // batches of 16 loads, added in order
                    float4 w[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (q0 + q < KS) w[q] = __ldcg(src + (q0 + q) * stride);
                    if (q0 == 0) v = w[0];
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (q0 + q < KS && q0 + q > 0) { v.x += w[q].x; v.y += w[q].y; v.z += w[q].z; v.w += w[q].w; }
                }
                *reinterpret_cast<float4 *>(S.L + tl * E + 4 * g) = v;
            }
        } else {
            for (int it = tid; it < CH * E; it += NT) {
                const int tl = it / E, e = it - tl * E, t = t0 + c0 + tl;
                if (t >= a.T) continue;
                float v = __ldcg(a.part + static_cast<size_t>(t) * E + e);
                for (int q = 1; q < KS; ++q) v += __ldcg(a.part + (static_cast<size_t>(q) * a.T + t) * E + e);
                S.L[tl * E + e] = v;
            }
        }
        for (int tl = tid; tl < CH; tl += NT) {
            const int t = t0 + c0 + tl;
            if (t >= a.T) continue;
            float n2 = 0.f;
            for (int q = 0; q < KS; ++q) n2 += __ldcg(a.xsq + static_cast<size_t>(q) * a.T + t);
            S.nxs[tl] = sqrtf(n2) * bd.infl;
        }
        __syncthreads();

        for (int tl = warp; tl < CH; tl += NW) {
            const int t = t0 + c0 + tl;
            if (t >= a.T) break;
            for (int e = lane; e < E; e += 32) S.sel[e] = S.L[tl * E + e];
            __syncwarp();
            uint32_t cand;
            int n_cand;
            int32_t *oi = a.topk_idx + static_cast<size_t>(t) * a.K;
            float *ow = a.topk_w + static_cast<size_t>(t) * a.K;
            bool every = false;
            uint32_t ck = kFullMask, ug = 0u;
            if (a.variant) {
                const int r = score_select_general(a, S.nxs[tl], S.nw, S.bias, bd.gam, S.sel,
                                                   S.bnd, S.sc, oi, ow, cand, n_cand, ck, ug,
                                                   lane);
                if (r > 0) continue;
                if (r < 0) {
                    every = true;
                    cand = all_experts(E, lane);
                    n_cand = E;
                }
            } else if (score_select(E, a.K, S.nxs[tl], S.nw, S.bias, bd.gam, S.sel, S.bnd, S.sc,
                                    oi, ow, cand, n_cand, lane)) {
                continue;
            }
            if (!every && n_cand < a.K) {   // non-finite scores: re-score every expert
                every = true;
                cand = all_experts(E, lane);
                n_cand = E;
            }
            // not certified: queue the candidates for the CTA-wide double-word refine
            int base = 0;
            if (lane == 0) base = atomicAdd(&s_npairs, n_cand);
            base = __shfl_sync(kFullMask, base, 0);
            if (base + n_cand <= a.max_pairs) {
                list_candidates(cand, E, S.p_e + base, lane);
                // default options: only candidates whose interval meets another's are
                // re-scored (p_tok < 0 marks the others, which keep their fp32 sel)
                const bool some = !a.variant && n_cand <= 32;
                const bool meets = some ? meets_another(S.p_e + base, n_cand, S.sel, S.bnd, lane) : true;
                for (int q = lane; q < n_cand; q += 32) {
                    const bool need = !some || meets;
                    S.p_tok[base + q] = need ? c0 + tl : -1 - (c0 + tl);
                    if (!need) S.p_val[base + q] = static_cast<double>(S.sel[S.p_e[base + q]]);
                }
                if (lane == 0) {
                    const int pi = atomicAdd(&s_npend, 1);
                    s_pend[5 * pi] = c0 + tl;
                    s_pend[5 * pi + 1] = base;
                    s_pend[5 * pi + 2] = every ? -n_cand : n_cand;   // < 0: every expert
                    s_pend[5 * pi + 3] = static_cast<int>(ck);
                    s_pend[5 * pi + 4] = static_cast<int>(ug);
                }
                __syncwarp();
                continue;
            }
            // list full (pathological ties): retire the reserved in-range slots, then
            // refine this token with the warp alone
            for (int q = base + lane; q < a.max_pairs; q += 32) S.p_e[q] = -1;
            __syncwarp();
            refine_token_warp(a, t, cand, S.ce, S.s64, S.ord, lane, every, ck, ug);
        }
    }
    __syncthreads();

    // CTA-wide refine of the queued tokens' (token, expert) pairs
    rescore_pairs(a, S.p_e, S.p_tok, min(s_npairs, a.max_pairs), t0, S.bias, S.need, S.dwp,
                  S.p_val, &s_nneed, warp, lane);
    for (int pi = warp; pi < s_npend; pi += NW) {
        const int tl = s_pend[5 * pi], first = s_pend[5 * pi + 1], cnt = s_pend[5 * pi + 2];
        const uint32_t ck = static_cast<uint32_t>(s_pend[5 * pi + 3]);
        const uint32_t ug = static_cast<uint32_t>(s_pend[5 * pi + 4]);
        const int t = t0 + tl;
        if (a.variant && cnt < 0)
            select_general64(a, S.p_e + first, S.p_val + first,
                             a.topk_idx + static_cast<size_t>(t) * a.K,
                             a.topk_w + static_cast<size_t>(t) * a.K, S.ord, lane);
        else if (a.variant)
            select_candidates64(a, S.p_e + first, S.p_val + first, cnt, ck, ug,
                                a.topk_idx + static_cast<size_t>(t) * a.K,
                                a.topk_w + static_cast<size_t>(t) * a.K, S.ord, lane);
        else
            select_refined(S.p_e + first, S.p_val + first, cnt < 0 ? -cnt : cnt, a.K, a.bias,
                           a.topk_idx + static_cast<size_t>(t) * a.K,
                           a.topk_w + static_cast<size_t>(t) * a.K, S.ord, lane);
    }
}

// ------------------------------------------- GEMM-only kernels + finaliser
template <class C>
__global__ void __launch_bounds__(NT_WS, 1) router_gemm_kernel(const RouterArgs a)
{
    pdl_wait();
    extern __shared__ __align__(16) unsigned char smem[];
    gemm_tile_ws<C>(a, smem);
}

// Shared-memory layout of the finalise launch: one CTA finalises up to NW consecutive
// tokens (one warp each for scoring and selection), then re-scores the uncertified
// candidates of all of them together.
struct FinCta {
    float *nw, *bias, *L, *bnd, *sc, *nxs;   // [E] x 2, [NW][E] x 3 (logits -> sel), [NW]
    int *ce, *ord;                     // [NW][E] (per-warp fallback), [NW][32]
    int *p_e, *p_tok, *need;           // refine list [MP] x 3
    double *p_val, *s64;               // [MP], [NW][E] (per-warp fallback)
    float2 *dwp;                       // [NW] partial double-word dot of each warp

    __host__ __device__ static int pairs(int E) { return E > 512 ? 1024 : 2048; }
    __device__ FinCta(unsigned char *smem, int E)
    {
        const int MP = pairs(E);
        float *f = reinterpret_cast<float *>(smem);
        dwp = reinterpret_cast<float2 *>(f); f += 2 * NW;   // (first: 8-byte aligned)
        nw = f; f += E;
        bias = f; f += E;
        L = f; f += NW * E;                                  // (16-byte aligned when E % 4 == 0)
        bnd = f; f += NW * E;
        sc = f; f += NW * E;
        nxs = f; f += NW;
        int *i = reinterpret_cast<int *>(f);
        ce = i; i += NW * E;
        ord = i; i += NW * 32;
        p_e = i; i += MP;
        p_tok = i; i += MP;
        need = i; i += MP;
        const uintptr_t d = (reinterpret_cast<uintptr_t>(i) + 7) & ~static_cast<uintptr_t>(7);
        p_val = reinterpret_cast<double *>(d);
        s64 = p_val + MP;
    }
    static size_t bytes(int E)
    {
        const size_t MP = pairs(E);
        return (2 * static_cast<size_t>(E) + 3 * NW * static_cast<size_t>(E) + NW + 2 * NW) * 4 +
               (static_cast<size_t>(NW) * E + NW * 32 + 3 * MP) * 4 + 8 +
               (MP + static_cast<size_t>(NW) * E) * 8;
    }
};

// Split-K sum, scoring, certified top-K and refine of `tpc` (1, 2, 4 or 8) consecutive
// tokens per CTA (the CTA's tokens lie in one token tile of TT tokens, whose gate-row norms
// it forms).  Small batches take one token per CTA: the partial sums are read by many SMs
// at once (one SM keeps only so many loads in flight), and the CTA's eight warps are free
// to split that token's re-scores among them.
//   1. The whole CTA sums the split-K partials of its tokens, every split's float4 loads
//      of an element in flight together, added in split order.
//   2. One warp per token scores it and takes the certified top-K; a token the bounds do
//      not certify queues its candidates in a CTA-wide list (default options: only those
//      whose interval meets another candidate's need re-scoring).
//   3. The CTA re-scores the listed (token, expert) pairs in double-word arithmetic; with
//      few pairs, each dot product is split over a group of warps (ranges of H merged in
//      rank order), so one re-score costs about one memory round trip.
//   4. One warp per queued token selects among its re-scored candidates.
__global__ void __launch_bounds__(NT) router_finalize_kernel(const RouterArgs a, int TT, int tpc)
{
    pdl_wait();
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_npairs, s_npend, s_nneed;
    __shared__ int s_pend[5 * NW];      // (token, first pair, pair count, ck, ug) to select
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = a.E, KS = a.KS, MP = FinCta::pairs(E);
    const int t0 = blockIdx.x * tpc;
    const int ntok = min(tpc, a.T - t0);
    FinCta S(smem, E);
    const Bounds bd(a.depth, KS, a.H);
    const int tt = t0 / TT;
    if (tid == 0) { s_npairs = 0; s_npend = 0; s_nneed = 0; }

    // ---- 1. gate-row norms, token norms and the logits of the CTA's tokens
    for (int e = tid; e < E; e += NT) {
        float n = 0.f;
        for (int q0 = 0; q0 < KS; q0 += 32) {   // up to 32 loads in flight, in split order
            float pn[32];
#pragma unroll
            for (int q = 0; q < 32; ++q)
                if (q0 + q < KS) pn[q] = __ldcg(a.wsq + (static_cast<size_t>(tt) * KS + q0 + q) * E + e);
            if (q0 == 0) n = pn[0];
#pragma unroll
            for (int q = 0; q < 32; ++q)
                if (q0 + q < KS && q0 + q > 0) n += pn[q];
        }
        S.nw[e] = sqrtf(n) * bd.infl;
        S.bias[e] = a.bias[e];
    }
    if (warp == NW - 1 && lane < ntok) {   // token norms: every split's load in flight
        float n2 = 0.f;
        for (int q0 = 0; q0 < KS; q0 += 32) {
            float pq[32];
#pragma unroll
            for (int q = 0; q < 32; ++q)
                if (q0 + q < KS) pq[q] = __ldcg(a.xsq + static_cast<size_t>(q0 + q) * a.T + t0 + lane);
#pragma unroll
            for (int q = 0; q < 32; ++q)
                if (q0 + q < KS) n2 += pq[q];
        }
        S.nxs[lane] = sqrtf(n2) * bd.infl;
    }
    if ((E & 3) == 0) {
        // The partials of split q for the CTA's tokens are one contiguous block of `items`
        // float4.  With few tokens per CTA the splits are divided among G thread groups
        // (every warp carries loads, at most 8 in flight per thread): group g sums its
        // consecutive splits in order, then the G group sums are added in group order --
        // a chain no deeper than KS, as the error bound assumes.
        const int items = ntok * (E / 4);
        int G = 1;
        while (E >= 128 && 2 * G * items <= NT && 2 * G <= KS && G < 8) G *= 2;   // (stage fits)
        const size_t stride4 = static_cast<size_t>(a.T) * E / 4;
        const float4 *base = reinterpret_cast<const float4 *>(a.part) + static_cast<size_t>(t0) * (E / 4);
        float4 *stage = reinterpret_cast<float4 *>(S.bnd);      // [G][items] (free until step 2)
        for (int it0 = 0; it0 < items; it0 += NT / G) {
            const int it = it0 + tid % (NT / G), g = tid / (NT / G);
            if (it < items) {
                const int qb = g * KS / G, qe = (g + 1) * KS / G;
                const float4 *src = base + it;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int q0 = qb; q0 < qe; q0 += 8) {     // 8 loads in flight, in split order
                    float4 w[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (q0 + q < qe) w[q] = __ldcg(src + static_cast<size_t>(q0 + q) * stride4);
                    if (q0 == qb) v = w[0];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (q0 + q < qe && q0 + q > qb) { v.x += w[q].x; v.y += w[q].y; v.z += w[q].z; v.w += w[q].w; }
                }
                if (G == 1) *reinterpret_cast<float4 *>(S.L + 4 * static_cast<size_t>(it)) = v;
                else stage[static_cast<size_t>(g) * (NT / G) + (it - it0)] = v;
            }
            if (G > 1) {
                __syncthreads();
                if (tid < NT / G && it < items) {
                    float4 v = stage[tid];
                    for (int h = 1; h < G; ++h) {
                        const float4 o = stage[static_cast<size_t>(h) * (NT / G) + tid];
                        v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
                    }
                    *reinterpret_cast<float4 *>(S.L + 4 * static_cast<size_t>(it)) = v;
                }
                __syncthreads();
            }
        }
    } else {
        for (int it = tid; it < ntok * E; it += NT) {
            const int tl = it / E, e = it - tl * E;
            const float *src = a.part + static_cast<size_t>(t0 + tl) * E + e;
            float v = __ldcg(src);
            for (int q = 1; q < KS; ++q) v += __ldcg(src + static_cast<size_t>(q) * a.T * E);
            S.L[it] = v;
        }
    }
    __syncthreads();

    // ---- 2. scoring (default options: every thread takes (token, expert) pairs), then one
    // warp per token: the certified top-K, else its candidates are queued
    if (!a.variant) {
        for (int i = tid; i < ntok * E; i += NT) {
            const int tl = i / E, e = i - tl * E;
            float sel, bnd, sc;
            score_expert(S.L[i], bd.gam * S.nxs[tl] * S.nw[e] + 1e-30f, S.bias[e], sel, bnd, sc);
            S.L[i] = sel;
            S.bnd[i] = bnd;
            S.sc[i] = sc;
        }
        __syncthreads();
    }
    if (warp < ntok) {
        const int t = t0 + warp;
        float *w_sel = S.L + static_cast<size_t>(warp) * E;
        float *w_bnd = S.bnd + static_cast<size_t>(warp) * E, *w_sc = S.sc + static_cast<size_t>(warp) * E;
        int32_t *oi = a.topk_idx + static_cast<size_t>(t) * a.K;
        float *ow = a.topk_w + static_cast<size_t>(t) * a.K;
        uint32_t cand = 0u, ck = kFullMask, ug = 0u;
        int n_cand = 0;
        bool every = false, done = false;
        if (a.variant) {
            const int r = score_select_general(a, S.nxs[warp], S.nw, S.bias, bd.gam, w_sel, w_bnd,
                                               w_sc, oi, ow, cand, n_cand, ck, ug, lane);
            done = r > 0;
            if (r < 0) every = true;
        } else {
            done = select_scored(E, a.K, w_sel, w_bnd, w_sc, oi, ow, cand, n_cand, lane);
        }
        if (!done && !every && n_cand < a.K) every = true;   // non-finite scores
        if (!done) {
            if (every) {
                cand = all_experts(E, lane);
                n_cand = E;
            }
            int base = 0;
            if (lane == 0) base = atomicAdd(&s_npairs, n_cand);
            base = __shfl_sync(kFullMask, base, 0);
            if (base + n_cand <= MP) {
                list_candidates(cand, E, S.p_e + base, lane);
                // default options: only candidates whose interval meets another's are
                // re-scored (p_tok < 0 marks the others, which keep their fp32 sel)
                const bool some = !a.variant && !every && n_cand <= 32;
                const bool meets = some ? meets_another(S.p_e + base, n_cand, w_sel, w_bnd, lane) : true;
                for (int q = lane; q < n_cand; q += 32) {
                    const bool need = !some || meets;
                    S.p_tok[base + q] = need ? warp : -1 - warp;
                    if (!need) S.p_val[base + q] = static_cast<double>(w_sel[S.p_e[base + q]]);
                }
                if (lane == 0) {
                    const int pi = atomicAdd(&s_npend, 1);
                    s_pend[5 * pi] = warp;
                    s_pend[5 * pi + 1] = base;
                    s_pend[5 * pi + 2] = every ? -n_cand : n_cand;   // < 0: every expert
                    s_pend[5 * pi + 3] = static_cast<int>(ck);
                    s_pend[5 * pi + 4] = static_cast<int>(ug);
                }
                __syncwarp();
            } else {
                // list full (pathological ties): retire the reserved in-range slots, then
                // refine this token with the warp alone
                for (int q = base + lane; q < MP; q += 32) S.p_e[q] = -1;
                __syncwarp();
                refine_token_warp(a, t, cand, S.ce + static_cast<size_t>(warp) * E,
                                  S.s64 + static_cast<size_t>(warp) * E, S.ord + warp * 32, lane,
                                  every, ck, ug);
            }
        }
    }
    __syncthreads();

    // ---- 3. the listed pairs re-scored by the whole CTA
    rescore_pairs(a, S.p_e, S.p_tok, min(s_npairs, MP), t0, S.bias, S.need, S.dwp, S.p_val,
                  &s_nneed, warp, lane);

    // ---- 4. selection among the re-scored candidates, one warp per queued token
    for (int pi = warp; pi < s_npend; pi += NW) {
        const int tl = s_pend[5 * pi], first = s_pend[5 * pi + 1], cnt = s_pend[5 * pi + 2];
        const uint32_t ck = static_cast<uint32_t>(s_pend[5 * pi + 3]);
        const uint32_t ug = static_cast<uint32_t>(s_pend[5 * pi + 4]);
        const int t = t0 + tl;
        int *ord = S.ord + warp * 32;
        if (a.variant && cnt < 0)
            select_general64(a, S.p_e + first, S.p_val + first,
                             a.topk_idx + static_cast<size_t>(t) * a.K,
                             a.topk_w + static_cast<size_t>(t) * a.K, ord, lane);
        else if (a.variant)
            select_candidates64(a, S.p_e + first, S.p_val + first, cnt, ck, ug,
                                a.topk_idx + static_cast<size_t>(t) * a.K,
                                a.topk_w + static_cast<size_t>(t) * a.K, ord, lane);
        else
            select_refined(S.p_e + first, S.p_val + first, cnt < 0 ? -cnt : cnt, a.K, S.bias,
                           a.topk_idx + static_cast<size_t>(t) * a.K,
                           a.topk_w + static_cast<size_t>(t) * a.K, ord, lane);
    }
}

size_t fused_smem(int TT, int TE, int E, int max_pairs)
{
    const size_t g = 2 * KST * static_cast<size_t>(TT + TE) * sizeof(float);
    const size_t f = FinSmem::bytes(E, max_pairs);
    return (g > f ? g : f) + 16;
}

size_t finalize_smem(int E) { return FinCta::bytes(E) + 16; }

}  // namespace

// Small-tile batches of 16 to 2048 tokens select in the finalise launch (1 to 8 tokens a
// CTA over the whole GPU) rather than in the last CTA of each 16-token tile: 71.6 -> 63.1
// us at 128 tokens, 6 us less from 16 to 2048 tokens; at 4096 the last-CTA selection is
// ahead (654 vs 662 us).
constexpr int kSplitMinTokens = 16, kSplitMaxTokens = 2048;
constexpr size_t kMaxSmemPerCta = 232448;   // dynamic shared memory a CTA may opt in to

RouterPlan router_plan(int T, int H, int E)
{
    RouterPlan p{};
    const bool small = T <= 4096;
    // the one-launch paths finalise in one CTA whose shared memory holds E-wide arrays per
    // warp: past what a CTA may hold (E above ~800) the batch takes the tile GEMM and the
    // finalise launch instead
    const bool fused_ok = fused_smem(SmallCfg::TT, SmallCfg::TE, E, 1024) <= kMaxSmemPerCta;
    p.gemv = 0;                                  // token batch of the tiny-batch path
    if (T <= GEMV_TMAX && fused_ok)
        for (p.gemv = 1; p.gemv < T; p.gemv <<= 1) {}
    p.TT = small ? SmallCfg::TT : LargeCfg::TT;
    p.TE = p.gemv ? GEMV_EPC : (small ? SmallCfg::TE : LargeCfg::TE);
    p.nTT = (T + p.TT - 1) / p.TT;
    p.nET = (E + p.TE - 1) / p.TE;
    p.S = H / KST;
    const int base = p.nTT * p.nET;
    const bool split = !p.gemv && small &&
                       ((T >= kSplitMinTokens && T <= kSplitMaxTokens) || !fused_ok);
    // resident CTAs per SM: 2 for the two-stage small tile, 1 for the warp-specialised ones
    const int target = (small && !split ? 2 : 1) * num_sms();
    if (p.gemv) {
        p.KS = 1;
        p.depth = ((H / 8 + GEMV_QW - 1) / GEMV_QW + 31) / 32 + 3 + 5 + 2 + 2;
    } else {
        // at most 32 stages per split keeps the summation depth (and the error bound) small
        p.KS = (p.S + 31) / 32;
        // (the finalise sums at most 32 splits in one batch of loads)
        if (p.KS > 32) p.KS = 32;
        // split tiles (16 to 2048 tokens, one CTA per SM): the split count with the least
        // modelled time, waves x (stages of a split + the per-CTA overhead, ~0.7 of a
        // stage, measured at the DeepSeek-V3 shape), from 64 stages a split down to 32
        // splits -- the finalise launch reads every split's partials with their loads in
        // flight together, so more splits cost it little.  Otherwise: doubled while the
        // grid stays below one wave.
        if (split) {
            long long best = -1;
            const int ks_hi = p.S < 32 ? p.S : 32;
            for (int ks = (p.S + 63) / 64; ks <= ks_hi; ++ks) {
                const long long waves = (static_cast<long long>(base) * ks + target - 1) / target;
                const long long cost = waves * (((p.S + ks - 1) / ks) * 11 + 8);
                if (best < 0 || cost < best) { best = cost; p.KS = ks; }
            }
        } else {
            while (p.KS * 2 <= p.S && p.KS * 2 <= 32 && base * p.KS < target) p.KS *= 2;
        }
        p.depth = KST + (p.S + p.KS - 1) / p.KS + p.KS + 2;
    }
    p.split = split ? 1 : 0;
    p.max_pairs = 1024;
    auto al = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    p.part_bytes = al(static_cast<size_t>(p.KS) * T * E * sizeof(float));
    p.xsq_bytes = al(static_cast<size_t>(p.KS) * T * sizeof(float));
    p.wsq_bytes = al(static_cast<size_t>(p.nTT) * p.KS * E * sizeof(float));
    p.cnt_bytes = al(static_cast<size_t>(p.nTT) * sizeof(unsigned));
    p.smem_bytes = !small ? ws_smem_bytes<LargeCfg>()
                 : p.split ? ws_smem_bytes<SmallWsCfg>()
                           : fused_smem(p.TT, p.TE, E, p.max_pairs);
    return p;
}

cudaError_t launch_router(const void *X, const void *Wg, const float *bias, int T, int H,
                          int E, int K, int32_t *topk_idx, float *topk_w,
                          const RouterPlan &plan, const RouterScratch &scr, int *status,
                          cudaStream_t s, const RoutingOpts *ro)
{
    RouterArgs a{};
    const RoutingOpts opts = ro ? *ro : RoutingOpts{};
    a.scoring = opts.scoring;
    a.n_group = opts.n_group;
    a.topk_group = opts.topk_group;
    a.group_top = opts.group_top;
    a.renorm = opts.renorm;
    a.variant = opts.is_default() ? 0 : 1;
    a.X = static_cast<const uint16_t *>(X);
    a.Wg = static_cast<const uint16_t *>(Wg);
    a.bias = bias;
    a.T = T; a.H = H; a.E = E; a.K = K; a.KS = plan.KS; a.S = plan.S;
    a.part = scr.part; a.xsq = scr.xsq; a.wsq = scr.wsq; a.cnt = scr.cnt;
    a.topk_idx = topk_idx; a.topk_w = topk_w; a.status = status;
    a.max_pairs = plan.max_pairs;
    a.depth = plan.depth;
    dim3 grid(plan.nET, plan.nTT, plan.KS);
    cudaError_t err;
    if (plan.split) {
        err = ensure_smem(reinterpret_cast<const void *>(router_gemm_kernel<SmallWsCfg>), plan.smem_bytes);
        if (err != cudaSuccess) return err;
        if ((err = launch_pdl(router_gemm_kernel<SmallWsCfg>, grid, dim3(NT_WS), plan.smem_bytes, s, 1, a)) != cudaSuccess)
            return err;
    } else if (plan.TT == SmallCfg::TT) {
        err = cudaMemsetAsync(scr.cnt, 0, static_cast<size_t>(plan.nTT) * sizeof(unsigned), s);
        if (err != cudaSuccess) return err;
        const void *fn;
        switch (plan.gemv) {
        case 1: fn = reinterpret_cast<const void *>(router_fused_kernel<SmallCfg, 1>); break;
        case 2: fn = reinterpret_cast<const void *>(router_fused_kernel<SmallCfg, 2>); break;
        case 4: fn = reinterpret_cast<const void *>(router_fused_kernel<SmallCfg, 4>); break;
        case 8: fn = reinterpret_cast<const void *>(router_fused_kernel<SmallCfg, 8>); break;
        default: fn = reinterpret_cast<const void *>(router_fused_kernel<SmallCfg, 0>); break;
        }
        err = ensure_smem(fn, plan.smem_bytes);
        if (err != cudaSuccess) return err;
        switch (plan.gemv) {
        case 1: return launch_pdl(router_fused_kernel<SmallCfg, 1>, grid, dim3(NT), plan.smem_bytes, s, 1, a);
        case 2: return launch_pdl(router_fused_kernel<SmallCfg, 2>, grid, dim3(NT), plan.smem_bytes, s, 1, a);
        case 4: return launch_pdl(router_fused_kernel<SmallCfg, 4>, grid, dim3(NT), plan.smem_bytes, s, 1, a);
        case 8: return launch_pdl(router_fused_kernel<SmallCfg, 8>, grid, dim3(NT), plan.smem_bytes, s, 1, a);
        default: return launch_pdl(router_fused_kernel<SmallCfg, 0>, grid, dim3(NT), plan.smem_bytes, s, 1, a);
        }
    } else {
        err = ensure_smem(reinterpret_cast<const void *>(router_gemm_kernel<LargeCfg>), plan.smem_bytes);
        if (err != cudaSuccess) return err;
        if ((err = launch_pdl(router_gemm_kernel<LargeCfg>, grid, dim3(NT_WS), plan.smem_bytes, s, 1, a)) != cudaSuccess)
            return err;
    }
    const size_t fs = finalize_smem(E);
    err = ensure_smem(reinterpret_cast<const void *>(router_finalize_kernel), fs);
    if (err != cudaSuccess) return err;
    // tokens per finalise CTA: the fewest that keep the grid within one CTA per SM (its
    // registers allow one resident CTA)
    const int sms = num_sms();
    const int tpc = T <= sms ? 1 : (T <= 2 * sms ? 2 : (T <= 4 * sms ? 4 : NW));
    return launch_pdl(router_finalize_kernel, dim3((T + tpc - 1) / tpc), dim3(NT), fs, s, 1, a,
                      plan.TT, tpc);
}

}  // namespace moe
