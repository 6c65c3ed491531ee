// ffn_tc.cu -- grouped SwiGLU expert FFN on the 5th-generation tensor cores (tcgen05 +
// TMEM), fed by TMA, persistent over a tile list built on the device from the per-expert
// row offsets.
//
// Method: "Lower latency and higher throughput with multi-node DeepSeek deployment",
// section "Roofline / GroupGEMM": g groups, group i has m_i tokens and computes
// [m_i, k] x [k, n]; decode is bound by the bytes of the activated experts, prefill by the
// tensor cores.  Section "Quantization": the expert activation is SiLU-and-multiply.
// Section "Cuda Graph" / "MoE Router": persistent kernels read the routing counts on the
// device instead of sizing work from buffer sizes.
//
// Formulation (swap-AB).  Each tile computes D[128 x n] = A[128 x K] * B[K x n] with the
// WEIGHTS as the M=128 operand and the TOKENS as the N operand, so a decode tile with a
// handful of tokens still uses the full M=128 MMA and the weights are streamed exactly
// once per tile:
//   up   : A rows 0..63  = W1[g][:, i0..i0+63]^T, rows 64..127 = W3[g][:, i0..i0+63]^T
//          (two TMA boxes of the [H, I] weight, so A is MN-major), B = token rows (K-major);
//          epilogue h[row, i] = silu(G) * U with G in TMEM lanes 0..63, U in lanes 64..127.
//   down : A rows = W2[g][:, h0..h0+127]^T (MN-major), B = rows of h; epilogue writes
//          Yp[row, h0..h0+127] (bf16) or fp32.
//
// Roles (192 threads, one CTA per SM): warp 0 = TMA producer, warp 1 = TMEM allocator and
// MMA issuer, warps 2..5 = epilogue (TMEM -> registers -> global).  A `stages`-deep
// shared-memory ring (full/empty mbarriers) decouples TMA from the MMAs; two TMEM
// accumulators decouple the MMAs of tile j+1 from the epilogue of tile j.
//
// CTA pairs.  Token tiles of 128 rows or more run on clusters of two CTAs that issue
// 2-SM MMAs (cta_group::2): one 256-row weight tile per pair, each CTA staging 128 weight
// rows and half of the token rows, the even CTA issuing the MMAs and owning the ring's
// full barriers (both CTAs' copies complete there), commits multicast to both CTAs.  Per
// SM this halves the token-tile bytes in shared memory and the L2 reads per flop.
//
// Tile list and schedule.  One launch holds the up-projection tiles, then the down-
// projection tiles of every problem.  Within each phase, groups that reuse a weight tile
// across several token tiles (tensor-bound) come first, groups with a single, at most
// half-full token tile (weight-streaming) after them, the two sequences interleaved in
// proportion.  Units claim tiles in list order from a global counter (dynamic schedule),
// so the token tiles that share a weight tile are in flight together and L2 serves the
// second read; a down tile waits (bounded) until the up tiles of its token tile have
// published their h rows.
//
// FP8 (ffn_kernel<false, true>).  Weights and activations arrive as E4M3 bytes with
// power-of-two block scales ("Lower latency and higher throughput...", Quantization: one
// scale per 128 x 128 weight tile, one per 128-element activation vector): the weights
// transposed to K-major rows ([g][n][k]), the activation rows with their scales in a
// transposed table ([k/128][rows], fp32 2^k).  A stage holds one 128-wide K block: the
// E4M3 weight tile and the token rows; the block's scales (the token rows' and the two
// weight boxes') go to a separate, deeper ring of small slots, so that a stage is free
// again as soon as its MMAs are done.  The tensor cores multiply the E4M3 bytes
// (tcgen05.mma kind::f8f6f4, both operands K-major) into a fresh fp32 partial in TMEM (up
// to eight partials in flight), and the epilogue adds each partial times the block's
// weight scale and token scale into accumulators held in registers ("promotion" per K
// block, taken in batches of partials); at the end of the tile it applies SwiGLU (up) or
// stores (down) as the bf16 kernel does.  Single-CTA tiles of at most 32 token rows
// (larger groups take several token tiles).  FP8 tiles are 256 weight rows, as two MMAs of
// M = 128 into two TMEM regions: an up tile covers 128 columns of I (its W1 rows in region
// 0, its W3 rows in region 1, so each epilogue thread holds both G and U of its column),
// a down tile 256 rows of H -- twice the weight bytes of a stage.
//
// Every wait is bounded (globaltimer): when one runs out the kernel records
// MOE_ERR_DEVICE_TIMEOUT in the status word, the other roles leave their loops, copies and
// MMAs in flight are drained with bounded waits, TMEM is freed and the kernel returns.
#include <cuda.h>

#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int BM = 128;                   // MMA M (weight rows)
constexpr int BK = 64;                    // K per stage = one 128-byte swizzle row of bf16
constexpr int A_BYTES = BM * BK * 2;      // 16 KB: two 64x64 boxes
constexpr int HALF_A = A_BYTES / 2;
constexpr int NUM_THREADS = 192;          // producer, MMA, 4 epilogue warps
constexpr int NUM_THREADS_FP8 = 224;      // FP8: + the scale producer warp
constexpr int BK8 = 128;                  // FP8: K per stage = one 128-byte row of E4M3
constexpr int A8_BYTES = BM * BK8;        // FP8: 16 KB, one 128-row region (two 64-row boxes)
constexpr int BN8_MAX = 32;               // FP8: token rows per tile (register accumulators)
constexpr int NPB_MAX = 8;                // FP8: TMEM partial buffers (2 regions x 32 columns each)
constexpr int SR = 32;                    // FP8: slots of the scale ring (one per K block)
constexpr int TSC = 128;                  // FP8: scale-table entries per box (H, I <= 16384)
constexpr int MAX_GROUPS = 1024;          // groups of one problem
constexpr int MAX_CG = 1040;              // groups of all problems of a launch
constexpr int CW = 32;                    // epilogue chunk: accumulator columns per TMEM load
constexpr int XCHG_FLOATS = 2 * CW * 64;  // double-buffered G exchange (up epilogue)
constexpr int PH_UP = 0, PH_DOWN = 1;
constexpr int TQ = 4;                     // depth of the ring that hands claimed tiles to the roles
constexpr int NT_BLOCK = 8;               // token tiles per block of a group's tile order
constexpr int MAX_STAGES = 8;       // deeper rings measured slower at decode (HBM-bound up projection)
constexpr int MAX_STAGES_FP8 = 8;   // FP8 (10 measured the same at decode)

struct ProbDev {
    const int32_t *offsets;  // [n_groups + 1] on the device, or nullptr (one dense group)
    int n_groups;
    int dense_rows;
    int rows;                // rows of the activation and output buffers (offsets' bound)
    int mt_up, mt_dn;        // weight tiles per token tile: up, down
    int kb_up, kb_dn;        // K blocks: H / 64, I / 64
    int I, H;                // row lengths of h (up output) and of the down output
    int out_fp32;
    void *h;                 // bf16 [rows, I]
    void *out;               // [rows, H] bf16 or fp32
    // FP8 weights: scale exponents per 128 x 128 tile, [groups][H/128][I/128] for W1 and W3,
    // [groups][I/128][H/128] for W2
    const int32_t *s1, *s3, *s2;
};

struct FfnArgs {
    CUtensorMap upA[2];      // per problem: W1
    CUtensorMap upA3[2];     // per problem: W3
    CUtensorMap upB[2];      // per problem: activation rows [rows, H]
    CUtensorMap dnA[2];      // per problem: W2
    CUtensorMap dnB[2];      // per problem: h [rows, I]
    CUtensorMap upS[2];      // FP8, per problem: activation scales [H/128, rows] (fp32)
    CUtensorMap dnS[2];      // FP8, per problem: h scales [I/128, rows] (fp32)
    ProbDev prob[2];
    int n_probs;
    int bn;                  // token tile: multiple of 16, <= 256
    int stages;
    int tmem_cols;
    int tab;                 // stride of the shared-memory group tables (>= groups + 1)
    unsigned *ready;         // per token tile: up-projection weight tiles finished
    unsigned *next_tile;     // tile counter of this launch (zero at launch)
    int *status;
    unsigned long long timeout_ns;
    int inject;              // 1: the producer never fills a stage (bounded-wait test)
    int phase_only;          // -1: up and down tiles; 0: only up tiles; 1: only down tiles
};

struct Tile {
    int ph, pi, g, cg, mt, row0, nvalid, nti;
};

// bar.red.and over the 128 epilogue threads: every thread gets the AND of `ok`.
__device__ __forceinline__ bool epi_all(bool ok)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.and.pred q, 2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(ok ? 1u : 0u)
        : "memory");
    return r != 0;
}

// sigmoid(g) = 1 / (1 + e^-g) from the hardware exp2 and reciprocal approximations (a few
// ulp in fp32; h is rounded to bf16 right after).  e^-g overflows to +inf for g < -88 and
// the reciprocal of +inf is 0, the limit.
__device__ __forceinline__ float fast_sigmoid(float g)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + __expf(-g)));
    return r;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}


template <bool PAIR, bool FP8>
__global__ void __launch_bounds__(FP8 ? NUM_THREADS_FP8 : NUM_THREADS, 1)
    ffn_kernel(const __grid_constant__ FfnArgs p)
{
    static_assert(!(PAIR && FP8), "FP8 tiles run on single CTAs");
    constexpr int NT = FP8 ? NUM_THREADS_FP8 : NUM_THREADS;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int bn = p.bn, S = p.stages, tab = p.tab;
    // FP8: partial buffers in TMEM (every K block's MMAs go to the next one), each two
    // regions of bn columns
    const uint32_t npb = FP8 ? static_cast<uint32_t>(p.tmem_cols / (2 * bn)) : 2u;
    const int bn_cta = PAIR ? bn / 2 : bn;    // token rows of B staged in this CTA
    // stage: weight tile (SW128) | token rows (SW128)
    const int b_off = FP8 ? 2 * A8_BYTES : A_BYTES;           // token rows within a stage
    const int stage_bytes = b_off + bn_cta * 128;
    unsigned char *stage_base = smem;
    // FP8 scale ring: per slot the token rows' scales of one K block (bn + 4 fp32, the copy
    // starting at a multiple of 4 rows) and the exponents of the stage's two weight boxes
    const int sl_ints = ((bn + 4) * 4 + 15) & ~15;            // byte offset of the exponents
    const int sl_bytes = FP8 ? ((sl_ints + 8 + 127) & ~127) : 0;
    unsigned char *sring = smem + static_cast<size_t>(S) * stage_bytes;
    float *xbuf = reinterpret_cast<float *>(sring + static_cast<size_t>(FP8 ? SR : 0) * sl_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(xbuf + (FP8 ? 0 : XCHG_FLOATS));   // (FP8: no exchange)
    uint64_t *empty = full + S;
    // accumulator handoff MMA -> epilogue: bf16 two per-tile buffers, FP8 npb per-K-block
    // partials
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + NPB_MAX;
    uint64_t *drain = tempty + NPB_MAX;
    uint64_t *tqf = drain + 1;                                // [TQ] tile slot written
    uint64_t *tqe = tqf + TQ;                                 // [TQ] tile slot read by all roles
    uint64_t *sfull = tqe + TQ;                               // FP8: [SR] scale slot written
    uint64_t *sempty = sfull + (FP8 ? SR : 0);                // FP8: [SR] scale slot read
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sempty + (FP8 ? SR : 0));
    static_assert(BK == 64, "the MMA issuer unrolls four K16 steps per stage");
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // groups of all problems, problem 0's first: first row, rows, the tile order, the tile
    // prefix of each phase over that order, and the token-tile prefix in group order
    int *n_used_s = reinterpret_cast<int *>(tmem_slot + 2);   // groups with rows
    int *n_heavy_s = reinterpret_cast<int *>(tmem_slot + 3);  // ... of which heavy
    int *gstart = reinterpret_cast<int *>(tmem_slot + 4);     // [tab]
    int *gm = gstart + tab;                                   // [tab]
    int *gord = gm + tab;                                     // [tab] group ids, tile order
    int *gpre_up = gord + tab;                                // [tab] up tiles before gord[k]
    int *gpre_dn = gpre_up + tab;                             // [tab] down tiles before gord[k]
    int *ntp = gpre_dn + tab;                                 // [tab] token tiles before group
    int *tq = ntp + tab;                                      // [TQ][8] claimed tiles

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t tmo = p.timeout_ns;
    // A CTA pair (cluster of two) computes one 256-row tile: the even CTA issues the MMAs
    // and owns the full/tempty barriers; each CTA stages half of A and half of B.
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        if (FP8)
            for (int r = 0; r < SR; ++r) {
                mbar_init(&sfull[r], 1);
                mbar_init(&sempty[r], 128);   // the epilogue threads
            }
        for (int b = 0; b < NPB_MAX; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], PAIR ? 256 : 128);
        }
        mbar_init(drain, 1);
        for (int q = 0; q < TQ; ++q) {
            mbar_init(&tqf[q], 1);
            // consumers of a slot: MMA and epilogue (and in a pair the odd CTA's producer
            // and epilogue, which read their copy of the slot; with FP8 the scale producer)
            mbar_init(&tqe[q], PAIR ? 4 : (FP8 ? 3 : 2));
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int pi = 0; pi < p.n_probs; ++pi) {
            prefetch_tmap(&p.upA[pi]);
            prefetch_tmap(&p.upA3[pi]);
            prefetch_tmap(&p.upB[pi]);
            prefetch_tmap(&p.dnA[pi]);
            prefetch_tmap(&p.dnB[pi]);
            if (FP8) {
                prefetch_tmap(&p.upS[pi]);
                prefetch_tmap(&p.dnS[pi]);
            }
        }
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(tmem_slot, static_cast<uint32_t>(p.tmem_cols));
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, static_cast<uint32_t>(p.tmem_cols));
            tmem_relinquish();
        }
    }
    // everything above overlaps the previous kernel's tail; the group offsets and the
    // activations are that kernel's (or an earlier one's) output
    pdl_wait();
    // group row offsets -> shared memory
    const int n0 = p.prob[0].n_groups;
    const int n_cg = n0 + (p.n_probs > 1 ? p.prob[1].n_groups : 0);
    // (offsets that are not non-decreasing within [0, rows] would send tiles past the
    // buffers: the launch then records MOE_ERR_INVALID_ARG and runs no tile)
    int bad = 0;
    for (int pi = 0; pi < p.n_probs; ++pi) {
        const ProbDev &P = p.prob[pi];
        const int base = pi ? n0 : 0;
        for (int g = tid; g < P.n_groups; g += NT) {
            const int a = P.offsets ? P.offsets[g] : 0;
            const int b = P.offsets ? P.offsets[g + 1] : P.dense_rows;
            bad |= a < 0 || b < a || b > P.rows;
            gstart[base + g] = a;
            gm[base + g] = b - a;
        }
    }
    if (__syncthreads_or(bad)) {
        for (int cg = tid; cg < n_cg; cg += NT) gm[cg] = 0;
        if (tid == 0) report(p.status, MOE_ERR_INVALID_ARG);
        __syncthreads();
    }
    // Tile order, per phase (all up-projection tiles, then all down-projection tiles).  A
    // group whose rows fit in one token tile at most half full is "light": its weights
    // are streamed from HBM for little arithmetic.  The other ("heavy") groups reuse each
    // weight tile across several token tiles and are bound by the tensor cores.  Heavy
    // groups come first, then light ones (each set in group order), and the two tile
    // sequences are interleaved in proportion, so that at any time some units stream
    // weights while the others compute.
    if (warp == 0) {
        int n = 0;
        for (int pass = 0; pass < 2; ++pass) {
            for (int c0 = 0; c0 < n_cg; c0 += 32) {
                const int cg = c0 + lane;
                bool sel = false;
                if (cg < n_cg) {
                    const int m = gm[cg];
                    const bool light = 2 * m <= bn;
                    sel = m > 0 && (pass == 0 ? !light : light);
                }
                const uint32_t bal = __ballot_sync(kFullMask, sel);
                if (sel) gord[n + __popc(bal & ((1u << lane) - 1u))] = cg;
                n += __popc(bal);
            }
            if (pass == 0 && lane == 0) *n_heavy_s = n;
        }
        __syncwarp();
        int run_up = 0, run_dn = 0;
        for (int k0 = 0; k0 < n; k0 += 32) {
            const int k = k0 + lane;
            int nu = 0, nd = 0;
            if (k < n) {
                const int cg = gord[k];
                const ProbDev &P = p.prob[cg >= n0 ? 1 : 0];
                const int ntn = (gm[cg] + bn - 1) / bn;
                nu = ntn * P.mt_up;
                nd = ntn * P.mt_dn;
            }
            int iu = nu, id = nd;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int vu = __shfl_up_sync(kFullMask, iu, off);
                const int vd = __shfl_up_sync(kFullMask, id, off);
                if (lane >= off) { iu += vu; id += vd; }
            }
            if (k < n) {
                gpre_up[k] = run_up + iu - nu;
                gpre_dn[k] = run_dn + id - nd;
            }
            run_up += __shfl_sync(kFullMask, iu, 31);
            run_dn += __shfl_sync(kFullMask, id, 31);
        }
        if (lane == 0) {
            gpre_up[n] = run_up;
            gpre_dn[n] = run_dn;
            *n_used_s = n;
        }
    } else if (warp == 1) {
        // token-tile prefix in group order: readiness counter of (group, token tile)
        int run = 0;
        for (int c0 = 0; c0 < n_cg; c0 += 32) {
            const int cg = c0 + lane;
            const int nt = cg < n_cg ? (gm[cg] + bn - 1) / bn : 0;
            int incl = nt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(kFullMask, incl, off);
                if (lane >= off) incl += v;
            }
            if (cg < n_cg) ntp[cg] = run + incl - nt;
            run += __shfl_sync(kFullMask, incl, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();   // the peer's barriers exist before any remote arrive or copy
    tc_fence_after();

    const uint32_t tmem_base = *tmem_slot;
    const int n_used = *n_used_s;
    const int n_heavy_groups = *n_heavy_s;
    const int n_up = gpre_up[n_used], n_dn = gpre_dn[n_used];
    const int n_tiles = n_up + n_dn;                         // up tiles, then down tiles
    // a launch may take only one phase: [t_begin, t_end) of the list
    const int t_begin = p.phase_only == 1 ? n_up : 0;
    const int t_end = p.phase_only == 0 ? n_up : n_tiles;
    const int heavy_up = gpre_up[n_heavy_groups], heavy_dn = gpre_dn[n_heavy_groups];
    const int light_up = n_up - heavy_up, light_dn = n_dn - heavy_dn;
    // Position t of a phase's interleaved order (N tiles, NL light) is a light tile when
    // floor(NL (t+1) / N) > floor(NL t / N); its index in the heavy-then-light order is
    // then NH + floor(NL t / N), otherwise t - floor(NL t / N).
    auto decode_at = [&](int t) -> Tile {
        const int ph = t >= n_up ? PH_DOWN : PH_UP;
        const int N = ph ? n_dn : n_up, NL = ph ? light_dn : light_up, NH = ph ? heavy_dn : heavy_up;
        const int *gpre = ph ? gpre_dn : gpre_up;
        const int tl = t - (ph ? n_up : 0);
        const int lt0 = static_cast<int>(static_cast<long long>(NL) * tl / N);
        const int lt1 = static_cast<int>(static_cast<long long>(NL) * (tl + 1) / N);
        const int v = lt1 > lt0 ? NH + lt0 : tl - lt0;
        int lo = 0, hi = n_used - 1;   // last k with gpre[k] <= v
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (gpre[mid] <= v) lo = mid; else hi = mid - 1;
        }
        const int cg = gord[lo];
        Tile T;
        T.ph = ph;
        T.pi = cg >= n0 ? 1 : 0;
        T.g = cg - (T.pi ? n0 : 0);
        T.cg = cg;
        const int m = gm[cg];
        const int ntn = (m + bn - 1) / bn;
        const int local = v - gpre[lo];
        // A group's tiles are taken in blocks of NT_BLOCK token tiles: for each block, every
        // weight tile in turn, the block's token tiles innermost.  The weight tile is then
        // shared by token tiles in flight together, and the block's token rows stay in L2
        // while the weight tiles pass (a group with many token tiles would otherwise re-read
        // all of its rows from HBM for every weight tile).
        const int mtn = ph ? p.prob[T.pi].mt_dn : p.prob[T.pi].mt_up;
        const int nb = local / (mtn * NT_BLOCK);
        const int rem = local - nb * (mtn * NT_BLOCK);
        const int width = min(NT_BLOCK, ntn - nb * NT_BLOCK);
        T.mt = rem / width;
        const int nt = nb * NT_BLOCK + (rem - T.mt * width);
        T.row0 = gstart[cg] + nt * bn;
        T.nvalid = min(bn, m - nt * bn);
        T.nti = ntp[cg] + nt;
        return T;
    };
    // Dynamic schedule: the producer of the even CTA claims the next tile of the list from
    // a global counter and hands it to the other roles -- and to the odd CTA of a pair --
    // through a TQ-slot ring (tqf: written, tqe: read by every consumer).  Tiles are thus
    // taken in list order by whichever unit is free, so the token tiles that share a weight
    // tile are in flight together (L2 serves the second read) and the tail stays balanced.
    // A tile with ph < 0 ends the list.
    auto slot_read = [&](int q) -> Tile {
        const int *e = tq + 8 * q;
        Tile T;
        T.ph = e[0]; T.pi = e[1]; T.g = e[2]; T.cg = e[3];
        T.mt = e[4]; T.row0 = e[5]; T.nvalid = e[6]; T.nti = e[7];
        return T;
    };
    // The even CTA's own roles arrive locally; the odd CTA's arrive on the even CTA's
    // barrier with release at cluster scope, so the even CTA's waits on tqe and tempty
    // acquire at cluster scope (the odd CTA's reads of its slot copy and of its tensor
    // memory are then ordered before the even CTA overwrites them).
    auto tqe_arrive = [&](int q) {
        if (PAIR && !leader) mbar_arrive_cluster(mapa_shared(smem_u32(&tqe[q]), 0));
        else mbar_arrive(&tqe[q]);
    };
    // MMA N: the valid rows rounded up to the instruction's granule (a pair splits N
    // evenly between its two CTAs, 16 rows each at least)
    auto n_mma_of = [&](const Tile &T) -> int {
        const int n = PAIR ? (T.nvalid + 31) & ~31 : (T.nvalid + 15) & ~15;
        return n < bn ? n : bn;
    };
    // this CTA's m-tile: a pair tile covers two single-CTA m-tiles
    auto mt_cta = [&](const Tile &T) -> int { return PAIR ? 2 * T.mt + static_cast<int>(rank) : T.mt; };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && !p.inject) {
            uint32_t it = 0;
            bool ok = true;
            uint32_t s = 0, ph = 0;
            unsigned char *a = stage_base;
            const uint32_t full_c0 = PAIR ? mapa_shared(smem_u32(full), 0) : 0u;   // even CTA's full[0]
            uint32_t qs = 0, qph = 0;
            // claim the next tile of the list and publish it to every role (and to the odd CTA)
            // FP8: the counter's next value is fetched one claim ahead, so the atomic's round
            // trip overlaps a tile's loads instead of stalling the ring at the tile boundary
            unsigned pend = FP8 ? atomicAdd(p.next_tile, 1u) : 0u;
            auto claim = [&](Tile &T) -> bool {
                if (!(PAIR ? mbar_wait_cluster(&tqe[qs], qph ^ 1u, abort_flag, p.status, tmo)
                           : mbar_wait(&tqe[qs], qph ^ 1u, abort_flag, p.status, tmo)))
                    return false;
                unsigned ticket;
                if (FP8) {
                    ticket = pend;
                    pend = atomicAdd(p.next_tile, 1u);
                } else {
                    ticket = atomicAdd(p.next_tile, 1u);
                }
                const int t = t_begin + static_cast<int>(ticket);
                if (t < t_end) {
                    T = decode_at(t);
                } else {
                    T = Tile{};
                    T.ph = -1;
                }
                const int vals[8] = {T.ph, T.pi, T.g, T.cg, T.mt, T.row0, T.nvalid, T.nti};
                int *e = tq + 8 * qs;
#pragma unroll
                for (int j = 0; j < 8; ++j) e[j] = vals[j];
                mbar_arrive(&tqf[qs]);
                if (PAIR) {
                    const uint32_t pe = mapa_shared(smem_u32(e), 1);
#pragma unroll
                    for (int j = 0; j < 8; ++j) st_shared_cluster(pe + 4u * j, vals[j]);
                    mbar_arrive_cluster(mapa_shared(smem_u32(&tqf[qs]), 1));
                }
                if (++qs == TQ) { qs = 0; qph ^= 1u; }
                return true;
            };
            Tile next_T{};
            bool have_next = false;
            while (ok) {
                Tile T;
                if (!PAIR || leader) {
                    if (have_next) {
                        T = next_T;
                        have_next = false;
                    } else if (!claim(T)) {
                        ok = false;
                        break;
                    }
                    // CTA pairs and FP8 tiles claim the following tile before this tile's
                    // loads are issued, so the global atomic, the decode (the hand-over to the
                    // odd CTA, the FP8 scale table) overlap them instead of stalling the ring
                    // at the tile boundary (bf16 single-CTA decode tiles measured better
                    // claiming one tile at a time)
                    if ((PAIR || FP8) && T.ph >= 0) {
                        if (!claim(next_T)) { ok = false; break; }
                        have_next = true;
                    }
                } else {
                    // odd CTA of a pair: take the even CTA's claim
                    if (!mbar_wait_cluster(&tqf[qs], qph, abort_flag, p.status, tmo)) { ok = false; break; }
                    T = slot_read(qs);
                    tqe_arrive(qs);
                    if (++qs == TQ) { qs = 0; qph ^= 1u; }
                }
                if (T.ph < 0) break;
                const ProbDev &P = p.prob[T.pi];
                const int mt = mt_cta(T);
                const bool up = T.ph == PH_UP;
                const CUtensorMap *mA = up ? &p.upA[T.pi] : &p.dnA[T.pi];
                const CUtensorMap *mA2 = up ? &p.upA3[T.pi] : &p.dnA[T.pi];
                const CUtensorMap *mB = up ? &p.upB[T.pi] : &p.dnB[T.pi];
                // two boxes of A (W1 | W3, or two 64-column halves of W2), one of B (this
                // CTA's token rows)
                const int a0 = up ? mt * 64 : mt * 128;
                const int a1 = up ? mt * 64 : mt * 128 + 64;
                const int a8 = up ? mt * 128 : mt * 256;   // FP8: the tile's first weight row
                const int brow = T.row0 + (PAIR && !leader ? n_mma_of(T) / 2 : 0);
                const int kblocks = up ? P.kb_up : P.kb_dn;
                if (!up && p.phase_only != 1) {
                    // the h rows of this token tile are complete once every up-projection
                    // weight tile of it has been stored (each CTA of a pair stores half); a
                    // launch of the down projections alone follows the up projections' launch
                    // on the stream, which already orders h before it
                    const unsigned need = static_cast<unsigned>(P.mt_up * (PAIR ? 2 : 1));
                    const unsigned *flag = p.ready + T.nti;
                    if (ld_acquire(flag) < need) {
                        const uint64_t t0 = globaltimer_ns();
                        while (ld_acquire(flag) < need) {
                            if (*abort_flag) { ok = false; break; }
                            if (globaltimer_ns() - t0 > tmo) {
                                *abort_flag = 1;
                                report(p.status, MOE_ERR_DEVICE_TIMEOUT);
                                ok = false;
                                break;
                            }
                            __nanosleep(128);
                        }
                        if (!ok) break;
                    }
                    fence_proxy_async_global();   // generic-proxy stores -> these TMA reads
                }
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status, tmo)) { ok = false; break; }
                    if (FP8) {
                        // four K-major E4M3 weight boxes (region 0: rows a8, a8 + 64 of W1 or
                        // W2; region 1: the same rows of W3, or rows a8 + 128, a8 + 192 of W2)
                        // and the token rows
                        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(2 * A8_BYTES + bn_cta * 128));
                        const int r1 = up ? a8 : a8 + 128;
                        tma_load_3d(a, mA, &full[s], kb * BK8, a8, T.g);
                        tma_load_3d(a + A8_BYTES / 2, mA, &full[s], kb * BK8, a8 + 64, T.g);
                        tma_load_3d(a + A8_BYTES, mA2, &full[s], kb * BK8, r1, T.g);
                        tma_load_3d(a + 3 * A8_BYTES / 2, mA2, &full[s], kb * BK8, r1 + 64, T.g);
                        tma_load_2d(a + b_off, mB, &full[s], kb * BK8, brow);
                    } else if (!PAIR) {
                        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(stage_bytes));
                        tma_load_3d(a, mA, &full[s], a0, kb * BK, T.g);
                        tma_load_3d(a + HALF_A, mA2, &full[s], a1, kb * BK, T.g);
                        tma_load_2d(a + A_BYTES, mB, &full[s], kb * BK, brow);
                    } else {
                        // both CTAs' copies complete on the even CTA's barrier, which
                        // expects the bytes of both
                        if (leader) mbar_arrive_expect_tx(&full[s], 2u * static_cast<uint32_t>(stage_bytes));
                        const uint32_t fb = full_c0 + 8u * s;
                        tma_load_3d_pair(a, mA, fb, a0, kb * BK, T.g);
                        tma_load_3d_pair(a + HALF_A, mA2, fb, a1, kb * BK, T.g);
                        tma_load_2d_pair(a + A_BYTES, mB, fb, kb * BK, brow);
                    }
                    if (++s == static_cast<uint32_t>(S)) { s = 0; ph ^= 1u; a = stage_base; } else { a += stage_bytes; }
                }
            }
            // every copy issued lands before the CTA can exit (a no-op wait in normal runs:
            // the MMA warp has already waited on each of these phases).  In a pair the
            // even CTA's barriers count the copies of both CTAs (with FP8 weights each CTA's
            // count its own).
            if (!PAIR || leader || FP8) {
                const uint32_t n = it < static_cast<uint32_t>(S) ? it : static_cast<uint32_t>(S);
                for (uint32_t j = it - n; j < it; ++j) {
                    int dummy_abort = 0;
                    mbar_wait(&full[j % S], (j / S) & 1u, &dummy_abort, nullptr, 20000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMA issuer
        if (lane == 0 && (!PAIR || leader)) {
            // The issuing thread's work per stage is kept to a few adds: one stage of MMAs
            // lasts only ~512 tensor-core cycles, and a longer dependent chain here (index
            // division, descriptor packing) leaves the tensor pipe idle between stages.
            const uint32_t ring0 = smem_u32(stage_base);
            // A: bf16 MN-major (LBO = the 64-column half), FP8 K-major (128-byte rows)
            const uint64_t adesc0 = FP8 ? smem_desc_sw128(ring0, 16, 1024) : smem_desc_sw128(ring0, HALF_A, 1024);
            const uint64_t bdesc0 = smem_desc_sw128(ring0 + b_off, 16, 1024);
            const uint32_t stage16 = static_cast<uint32_t>(stage_bytes) >> 4;  // descriptor units
            // per K step: bf16 K16 = +2048 B along A (MN-major), +32 B along B; FP8 K32 =
            // +32 B along both
            constexpr uint32_t ASTEP = FP8 ? 2u : 128u;
            uint32_t s = 0, ph = 0, soff = 0, tc = 0;
            uint32_t pb = 0, pph = 0;                   // FP8: partial buffer
            bool ok = true;
            uint32_t qs = 0, qph = 0;
            for (;; ++tc) {
                if (!mbar_wait(&tqf[qs], qph, abort_flag, p.status, tmo)) { ok = false; break; }
                const Tile T = slot_read(qs);
                tqe_arrive(qs);
                if (++qs == TQ) { qs = 0; qph ^= 1u; }
                if (T.ph < 0) break;
                const ProbDev &P = p.prob[T.pi];
                const uint32_t b = tc & 1u, tph = (tc >> 1) & 1u;
                if (!FP8) {
                    if (!(PAIR ? mbar_wait_cluster(&tempty[b], tph ^ 1u, abort_flag, p.status, tmo)
                               : mbar_wait(&tempty[b], tph ^ 1u, abort_flag, p.status, tmo))) { ok = false; break; }
                    tc_fence_after();
                }
                const int n_mma = n_mma_of(T);
                const uint32_t idesc = FP8 ? idesc_e4m3_f32(BM, static_cast<uint32_t>(n_mma))
                                           : idesc_bf16_f32(PAIR ? 2 * BM : BM, static_cast<uint32_t>(n_mma), true, false);
                const int kblocks = T.ph == PH_UP ? P.kb_up : P.kb_dn;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(&full[s], ph, abort_flag, p.status, tmo)) { ok = false; break; }
                    // FP8: every K block goes to a fresh partial the epilogue has emptied
                    if (FP8 && !mbar_wait(&tempty[pb], pph ^ 1u, abort_flag, p.status, tmo)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = adesc0 + soff, bd = bdesc0 + soff;
                    if (FP8) {
                        // region 0 (A rows 0..127) and region 1 (A rows 128..255, 16 KB on)
                        const uint32_t d = tmem_base + pb * 2u * static_cast<uint32_t>(bn);
                        const uint32_t d1 = d + static_cast<uint32_t>(bn);
                        constexpr uint64_t AR1 = static_cast<uint64_t>(A8_BYTES) >> 4;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            tc_mma_f8(d, ad + k * ASTEP, bd + 2 * k, idesc, k ? 1u : 0u);
                            tc_mma_f8(d1, ad + AR1 + k * ASTEP, bd + 2 * k, idesc, k ? 1u : 0u);
                        }
                        tc_commit(&empty[s]);
                        tc_commit(&tfull[pb]);
                        if (++pb == npb) { pb = 0; pph ^= 1u; }
                    } else if (PAIR) {
                        const uint32_t d_tmem = tmem_base + b * static_cast<uint32_t>(bn);
                        tc_mma_bf16_pair(d_tmem, ad, bd, idesc, kb != 0 ? 1u : 0u);
                        tc_mma_bf16_pair(d_tmem, ad + ASTEP, bd + 2, idesc, 1u);
                        tc_mma_bf16_pair(d_tmem, ad + 2 * ASTEP, bd + 4, idesc, 1u);
                        tc_mma_bf16_pair(d_tmem, ad + 3 * ASTEP, bd + 6, idesc, 1u);
                        tc_commit_pair_mc(&empty[s], 3);
                    } else {
                        const uint32_t d_tmem = tmem_base + b * static_cast<uint32_t>(bn);
                        tc_mma_bf16(d_tmem, ad, bd, idesc, kb != 0 ? 1u : 0u);
                        tc_mma_bf16(d_tmem, ad + ASTEP, bd + 2, idesc, 1u);
                        tc_mma_bf16(d_tmem, ad + 2 * ASTEP, bd + 4, idesc, 1u);
                        tc_mma_bf16(d_tmem, ad + 3 * ASTEP, bd + 6, idesc, 1u);
                        tc_commit(&empty[s]);
                    }
                    if (++s == static_cast<uint32_t>(S)) { s = 0; ph ^= 1u; soff = 0; } else { soff += stage16; }
                }
                if (!ok) break;
                if (!FP8) {
                    if (PAIR) tc_commit_pair_mc(&tfull[b], 3); else tc_commit(&tfull[b]);
                }
            }
            // drain: every MMA issued by this thread has completed before TMEM is freed
            if (PAIR) tc_commit_pair_mc(drain, 1); else tc_commit(drain);
            int dummy_abort = 0;
            mbar_wait(drain, 0, &dummy_abort, nullptr, 20000000ull);
        }
    } else if (FP8 && warp == 6) {
        // ------------------------------------------------------- FP8 scale producer
        // For every K block of every tile, in the order of the other roles: the token rows'
        // scales (a TMA copy from row0 rounded down to a multiple of 4 rows: a TMA copy's
        // innermost coordinate must be 16-byte aligned) and the exponents of the tile's two
        // weight boxes (asynchronous 4-byte copies whose completion the slot barrier
        // tracks) into the next slot of the scale ring.  Kept off the TMA producer's thread,
        // whose per-stage work sets the pace of the weight stream.
        if (lane == 0 && !p.inject) {
            uint32_t r = 0, rph = 0, n_sc = 0, qs = 0, qph = 0;
            bool ok = true;
            while (ok) {
                if (!mbar_wait(&tqf[qs], qph, abort_flag, p.status, tmo)) break;
                const Tile T = slot_read(qs);
                tqe_arrive(qs);
                if (++qs == TQ) { qs = 0; qph ^= 1u; }
                if (T.ph < 0) break;
                const ProbDev &P = p.prob[T.pi];
                const bool up = T.ph == PH_UP;
                // the two regions' first weight rows: up, the tile's 128 columns of W1 and
                // of W3; down, two 128-row halves of the tile's 256 rows of W2
                const int a0 = up ? T.mt * 128 : T.mt * 256, a1 = up ? T.mt * 128 : T.mt * 256 + 128;
                // the regions' exponents, one per K block (row stride nc of the
                // [g][K/128][N/128] table; a region past the last weight column reads zeros:
                // any tile's scale does, so its index is clamped)
                const int nc = (up ? P.I : P.H) / 128, nr = (up ? P.H : P.I) / 128;
                const int32_t *src[2];
                for (int box = 0; box < 2; ++box) {
                    const int c = min((box ? a1 : a0) / 128, nc - 1);
                    src[box] = (up ? (box ? P.s3 : P.s1) : P.s2) + static_cast<size_t>(T.g) * nr * nc + c;
                }
                const CUtensorMap *mS = up ? &p.upS[T.pi] : &p.dnS[T.pi];
                const int kblocks = up ? P.kb_up : P.kb_dn;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(&sempty[r], rph ^ 1u, abort_flag, p.status, tmo)) { ok = false; break; }
                    unsigned char *sl = sring + static_cast<size_t>(r) * sl_bytes;
                    const uint32_t ex = smem_u32(sl + sl_ints);
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;"
                                 ::"r"(ex), "l"(reinterpret_cast<uint64_t>(src[0] + static_cast<size_t>(kb) * nc))
                                 : "memory");
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;"
                                 ::"r"(ex + 4u), "l"(reinterpret_cast<uint64_t>(src[1] + static_cast<size_t>(kb) * nc))
                                 : "memory");
                    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];"
                                 ::"r"(smem_u32(&sfull[r])) : "memory");
                    mbar_arrive_expect_tx(&sfull[r], static_cast<uint32_t>((bn + 4) * 4));
                    tma_load_2d(sl, mS, &sfull[r], T.row0 & ~3, kb);
                    ++n_sc;
                    if (++r == static_cast<uint32_t>(SR)) { r = 0; rph ^= 1u; }
                }
            }
            // every copy issued lands before the CTA can exit
            asm volatile("cp.async.wait_all;" ::: "memory");
            const uint32_t n = n_sc < static_cast<uint32_t>(SR) ? n_sc : static_cast<uint32_t>(SR);
            for (uint32_t j = n_sc - n; j < n_sc; ++j) {
                int dummy_abort = 0;
                mbar_wait(&sfull[j % SR], (j / SR) & 1u, &dummy_abort, nullptr, 20000000ull);
            }
        }
    } else {
        // ----------------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        uint32_t tc = 0, cc = 0;
        uint32_t qs = 0, qph = 0;
        uint32_t es = 0, eph = 0, epb = 0, epph = 0;   // FP8: scale slot and partial buffer
        for (;; ++tc) {
            const bool okq = (PAIR && !leader)
                                 ? mbar_wait_cluster(&tqf[qs], qph, abort_flag, p.status, tmo)
                                 : mbar_wait(&tqf[qs], qph, abort_flag, p.status, tmo);
            if (!epi_all(okq)) break;
            const Tile T = slot_read(qs);
            named_bar_sync(4, 128);                 // every epilogue thread has read the slot
            if (warp == 2 && lane == 0) tqe_arrive(qs);
            if (++qs == TQ) { qs = 0; qph ^= 1u; }
            if (T.ph < 0) break;
            const ProbDev &P = p.prob[T.pi];
            const uint32_t b = tc & 1u, tph = (tc >> 1) & 1u;
            const int nchunks = (T.nvalid + CW - 1) / CW;
            const int mt = mt_cta(T);
            // 32 lanes x 16 or 32 columns of TMEM (a 16-row tile has 16 columns per buffer)
            auto tmem_cols = [&](uint32_t taddr, float (&v)[CW]) {
                __syncwarp();
                if (bn >= CW) {
                    tmem_ld32(taddr, v);
                } else {
                    float h[16];
                    tmem_ld16(taddr, h);
#pragma unroll
                    for (int j = 0; j < 16; ++j) { v[j] = h[j]; v[j + 16] = 0.f; }
                }
            };
            // FP8: the tile's accumulators, region r (0: W1 / first W2 half, 1: W3 / second
            // W2 half) x token column j (at most 32)
            float acc[2][CW];
            if (FP8) {
                // promotion: every K block's partial times 2^(weight tile exponent) times
                // the token row's 2^(exponent), added in K-block order.  The partials are
                // taken in batches of 128 TMEM columns (2 K blocks x 2 regions of 32 rows, or
                // 4 x 2 of 16): one round of waits, one barrier and one load latency per batch.
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int j = 0; j < CW; ++j) acc[r][j] = 0.f;
                const int kblocks = T.ph == PH_UP ? P.kb_up : P.kb_dn;
                const int per_batch = bn == 16 ? 4 : 2;              // K blocks a batch
                const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
                bool got_all = true;
                int kb0 = 0;
                while (kb0 < kblocks) {
                    // K blocks of this batch: within the tile and the partial ring
                    int nb = kblocks - kb0;
                    if (nb > per_batch) nb = per_batch;
                    if (nb > static_cast<int>(npb - epb)) nb = static_cast<int>(npb - epb);
                    bool got = true;
                    {
                        uint32_t si = es, phi = eph;
                        for (int i = 0; i < nb; ++i) {
                            got = got && mbar_wait(&sfull[si], phi, abort_flag, p.status, tmo) &&
                                  mbar_wait(&tfull[epb + i], epph, abort_flag, p.status, tmo);
                            if (++si == static_cast<uint32_t>(SR)) { si = 0; phi ^= 1u; }
                        }
                    }
                    if (!epi_all(got)) { got_all = false; break; }
                    tc_fence_after();
                    __syncwarp();
                    // K block i, region r of the batch: columns (2 i + r) bn on from the first
                    // partial
                    float v[128];
                    const uint32_t pb0 = tmem_base + lane_off + epb * 2u * static_cast<uint32_t>(bn);
                    if (bn == 16) {
                        uint32_t ad[8];
#pragma unroll
                        for (int l = 0; l < 8; ++l) ad[l] = pb0 + 16u * static_cast<uint32_t>((l >> 1) < nb ? l : 0);
                        tmem_ld16x8(ad, v);
                    } else {
                        uint32_t ad[4];
#pragma unroll
                        for (int l = 0; l < 4; ++l) ad[l] = pb0 + 32u * static_cast<uint32_t>((l >> 1) < nb ? l : 0);
                        tmem_ld32x4(ad[0], ad[1], ad[2], ad[3], v);
                    }
                    // the scales of K block i sit in scale slot es + i
                    auto block_scales = [&](int i, float &sw0, float &sw1, const float *&xs) {
                        uint32_t si = es + static_cast<uint32_t>(i);
                        if (si >= static_cast<uint32_t>(SR)) si -= static_cast<uint32_t>(SR);
                        const unsigned char *sl = sring + static_cast<size_t>(si) * sl_bytes;
                        const int *ex = reinterpret_cast<const int *>(sl + sl_ints);
                        sw0 = pow2f(ex[0]);
                        sw1 = pow2f(ex[1]);
                        xs = reinterpret_cast<const float *>(sl) + (T.row0 & 3);
                    };
                    if (bn == 16) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            if (i < nb) {
                                float sw0, sw1;
                                const float *xs;
                                block_scales(i, sw0, sw1, xs);
#pragma unroll
                                for (int j = 0; j < 16; ++j) {
                                    acc[0][j] = fmaf(v[32 * i + j], sw0 * xs[j], acc[0][j]);
                                    acc[1][j] = fmaf(v[32 * i + 16 + j], sw1 * xs[j], acc[1][j]);
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            if (i < nb) {
                                float sw0, sw1;
                                const float *xs;
                                block_scales(i, sw0, sw1, xs);
#pragma unroll
                                for (int j = 0; j < CW; ++j) {
                                    acc[0][j] = fmaf(v[64 * i + j], sw0 * xs[j], acc[0][j]);
                                    acc[1][j] = fmaf(v[64 * i + 32 + j], sw1 * xs[j], acc[1][j]);
                                }
                            }
                        }
                    }
                    // release the batch's partials and scale slots
                    tc_fence_before();
                    for (int i = 0; i < nb; ++i) {
                        mbar_arrive(&tempty[epb + i]);
                        mbar_arrive(&sempty[es]);
                        if (++es == static_cast<uint32_t>(SR)) { es = 0; eph ^= 1u; }
                    }
                    epb += static_cast<uint32_t>(nb);
                    if (epb == npb) { epb = 0; epph ^= 1u; }
                    kb0 += nb;
                }
                if (!got_all) break;
                // output: up, h = silu(G) * U of column i for every token (G and U of the
                // same column sit in the same thread); down, the thread's two rows of Yp
                if (T.ph == PH_UP) {
                    const int i = T.mt * 128 + 32 * q + lane;
                    if (i < P.I) {
                        uint16_t *out = static_cast<uint16_t *>(P.h);
#pragma unroll
                        for (int j = 0; j < CW; ++j) {
                            if (j < T.nvalid) {
                                const float g = acc[0][j];
                                out[static_cast<size_t>(T.row0 + j) * P.I + i] = f32_to_bf16_rn(g * fast_sigmoid(g) * acc[1][j]);
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int col = T.mt * 256 + 128 * r + 32 * q + lane;
                        if (col >= P.H) continue;
#pragma unroll
                        for (int j = 0; j < CW; ++j) {
                            if (j >= T.nvalid) continue;
                            const size_t o = static_cast<size_t>(T.row0 + j) * P.H + col;
                            if (P.out_fp32) static_cast<float *>(P.out)[o] = acc[r][j];
                            else static_cast<uint16_t *>(P.out)[o] = f32_to_bf16_rn(acc[r][j]);
                        }
                    }
                }
                continue;   // (FP8 tiles have no per-tile TMEM accumulator to release)
            } else {
                const bool ok = mbar_wait(&tfull[b], tph, abort_flag, p.status, tmo);
                if (!epi_all(ok)) break;
                tc_fence_after();
            }
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * static_cast<uint32_t>(bn);
            // one chunk = CW token columns of this warp's 32 accumulator rows
            auto load_chunk = [&](int c, float (&v)[CW]) { tmem_cols(tbase + CW * c, v); };
            if (T.ph == PH_UP) {
                // G (W1 rows) sits in lanes 0..63 (quarters 0, 1), U (W3 rows) in lanes
                // 64..127 (quarters 2, 3): the G warps hand their values over through shared
                // memory and the U warps -- which share no SM sub-partition with the
                // producer and MMA warps -- compute h = silu(G) * U and store it
                const int i = mt * 64 + (q & 1) * 32 + lane;
                const bool col_ok = i < P.I;
                uint16_t *out = static_cast<uint16_t *>(P.h);
                for (int c = 0; c < nchunks; ++c, ++cc) {
                    float v[CW];
                    load_chunk(c, v);
                    float *xb = xbuf + (cc & 1u) * (CW * 64);
                    if (q < 2) {
#pragma unroll
                        for (int j = 0; j < CW; ++j) xb[j * 64 + q * 32 + lane] = v[j];
                    }
                    named_bar_sync(1, 128);
                    if (q >= 2 && col_ok) {
#pragma unroll
                        for (int j = 0; j < CW; ++j) {
                            const int n = CW * c + j;
                            if (n < T.nvalid) {
                                const float g = xb[j * 64 + (q - 2) * 32 + lane];
                                const float h = g * fast_sigmoid(g) * v[j];
                                out[static_cast<size_t>(T.row0 + n) * P.I + i] = f32_to_bf16_rn(h);
                            }
                        }
                    }
                }
                // publish: this CTA's columns of the token tile are in h (generic-proxy
                // stores, read later by other SMs' TMA).  A launch of the up projections
                // alone is followed on the stream by the launch that reads h, which orders
                // the stores without fences or counters.
                if (p.phase_only != 0) {
                    fence_proxy_async_global();
                    __threadfence();
                    named_bar_sync(3, 128);
                    if (warp == 2 && lane == 0) atomicAdd(p.ready + T.nti, 1u);
                }
            } else {
                const int col = mt * 128 + q * 32 + lane;
                const bool col_ok = col < P.H;
                for (int c = 0; c < nchunks; ++c) {
                    float v[CW];
                    load_chunk(c, v);
                    if (col_ok) {
                        if (P.out_fp32) {
                            float *out = static_cast<float *>(P.out);
#pragma unroll
                            for (int j = 0; j < CW; ++j) {
                                const int n = CW * c + j;
                                if (n < T.nvalid) out[static_cast<size_t>(T.row0 + n) * P.H + col] = v[j];
                            }
                        } else {
                            uint16_t *out = static_cast<uint16_t *>(P.out);
#pragma unroll
                            for (int j = 0; j < CW; ++j) {
                                const int n = CW * c + j;
                                if (n < T.nvalid)
                                    out[static_cast<size_t>(T.row0 + n) * P.H + col] = f32_to_bf16_rn(v[j]);
                            }
                        }
                    }
                }
            }
            if (!FP8) {
                tc_fence_before();
                if (PAIR && !leader)
                    mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[b]), 0));
                else
                    mbar_arrive(&tempty[b]);
            }
        }
    }

    tc_fence_before();
    __syncwarp();
    __syncthreads();
    // neither CTA of a pair leaves (or frees tensor memory) while the other may still
    // signal its barriers or the even CTA's MMAs may still write its tensor memory
    if (PAIR) cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, static_cast<uint32_t>(p.tmem_cols));
        else
            tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));
    }
}

// ------------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    // looked up once (a function-local static is initialised once, even when several host
    // threads make their first calls together)
    static const EncodeTiledFn fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

// 3-D bf16 weight tensor [n_groups][rows][cols] (cols contiguous), 64 x 64 boxes in the
// 128-byte swizzle the MMA reads (MN-major operand).
bool encode_weight(CUtensorMap *m, const void *base, int n_groups, int rows, int cols)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(n_groups)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                             static_cast<cuuint64_t>(cols) * rows * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D E4M3 weight tensor [n_groups][n][k] (k contiguous: K-major rows), boxes of 128 k x 64
// rows in the 128-byte swizzle.
bool encode_weight8(CUtensorMap *m, const void *base, int n_groups, int n, int k)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(n),
                          static_cast<cuuint64_t>(n_groups)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(k) * n};
    cuuint32_t box[3] = {128, 64, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D E4M3 activation rows [rows][k], boxes of 128 k x box_rows rows (128-byte swizzle).
bool encode_act8(CUtensorMap *m, const void *base, int rows, int k, int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(k)};
    cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp32 scale table [blocks][pitch] (rows valid of each pitch), boxes of box_rows x 1.
bool encode_scales(CUtensorMap *m, const float *base, int rows, long long pitch, int blocks,
                   int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(blocks)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 activation tensor [rows][cols], boxes of 64 columns x box_rows rows.
bool encode_act(CUtensorMap *m, const void *base, int rows, int cols, int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token tile N: large enough that the busiest expert of a typical batch still fits in one
// tile (its weight tile is then streamed once), given only the mean rows per group.  The
// routing is skewed (the busiest of ~150 active experts holds ~5x the mean at T=128), so
// the tile covers 6x the mean.  The MMA's N is trimmed per tile to the valid rows anyway.
int pick_bn(int avg_rows)
{
    const long long want = 6ll * avg_rows;
    int bn = 16;
    while (bn < 256 && bn < want) bn <<= 1;
    return bn;
}

size_t ffn_smem_bytes(int bn_cta, int stages, int tab, bool fp8)
{
    const size_t stage = static_cast<size_t>(fp8 ? 2 * A8_BYTES : A_BYTES) + bn_cta * 128;
    const size_t slot = ((((bn_cta + 4) * 4 + 15) & ~static_cast<size_t>(15)) + 8 + 127) & ~static_cast<size_t>(127);
    return 1024 + stages * stage + (fp8 ? SR * slot : XCHG_FLOATS * 4) +
           (2 * stages + 2 * NPB_MAX + 1 + 2 * TQ) * 8 + (fp8 ? 2 * SR * 8 : 0) + 16 +
           (6 * static_cast<size_t>(tab) + 8 * TQ) * 4;
}

int pick_stages(int bn_cta, int tab, bool fp8)
{
    const size_t cap = 232448;   // max dynamic shared memory per block on sm_100/sm_103
    int s = fp8 ? MAX_STAGES_FP8 : MAX_STAGES;
    while (s > 2 && ffn_smem_bytes(bn_cta, s, tab, fp8) > cap) --s;
    return s;
}

// Token tiles of at least this many rows run on CTA pairs (256-row weight tiles, 2-SM
// MMA): per SM the pair halves the B tile held in shared memory and read by the tensor
// core, and halves the activation traffic from L2 per flop.
constexpr int PAIR_MIN_BN = 128;
int g_variant = 0;   // 0 automatic, 1 single CTA, 2 CTA pair

}  // namespace

void set_ffn_variant(int v) { g_variant = v; }

size_t ffn_ready_slots(long long rows, int n_groups)
{
    // token tiles are at least 16 rows: sum over groups of ceil(m / 16) <= rows / 16 + groups
    return static_cast<size_t>(rows / 16 + n_groups + 2);
}

cudaError_t launch_ffn(const FfnProblem *probs, int n_probs, int H, const int *I_pp,
                       int token_hint, unsigned *ready, bool ready_zeroed, int *status, cudaStream_t s,
                       unsigned long long timeout_ns, int inject, cudaEvent_t mid_event,
                       int phase_only, int max_ctas)
{
    if (n_probs < 1 || n_probs > 2 || !ready || phase_only < -1 || phase_only > 1)
        return cudaErrorInvalidValue;
    int n_cg = 0;
    long long rows_total = 0;
    const bool fp8 = probs[0].fp8 != 0;
    for (int pi = 0; pi < n_probs; ++pi) {
        if (probs[pi].n_groups < 1 || probs[pi].n_groups > MAX_GROUPS) return cudaErrorInvalidValue;
        if ((probs[pi].fp8 != 0) != fp8) return cudaErrorInvalidValue;
        if (fp8 && (!probs[pi].S1 || !probs[pi].S3 || !probs[pi].S2 || !probs[pi].act_s ||
                    !probs[pi].h8 || !probs[pi].h_s || H % 128 || I_pp[pi] % 128 ||
                    H > 128 * TSC || I_pp[pi] > 128 * TSC))
            return cudaErrorInvalidValue;
        n_cg += probs[pi].n_groups;
        rows_total += probs[pi].rows;
    }
    if (n_cg > MAX_CG) return cudaErrorInvalidValue;
    int bn = pick_bn(token_hint);
    if (fp8 && bn > BN8_MAX) bn = BN8_MAX;     // FP8: register accumulators, single CTAs
    bool pair = !fp8 && (g_variant == 2 || (g_variant == 0 && bn >= PAIR_MIN_BN));
    if (pair && bn < 32) bn = 32;           // 16 token rows per CTA at least
    const int bn_cta = pair ? bn / 2 : bn;
    const int tab = (n_cg + 1 + 3) & ~3;
    const int stages = pick_stages(bn_cta, tab, fp8);
    const size_t smem = ffn_smem_bytes(bn_cta, stages, tab, fp8);
    // TMEM columns: two accumulators of bn columns; FP8: NPB_MAX partials of two regions
    // of bn columns (at most 512)
    int tcols = 32;
    while (tcols < (fp8 ? 2 * NPB_MAX : 2) * bn && tcols < 512) tcols <<= 1;
    const int m_up = pair ? 128 : 64;      // weight columns of one tile
    const int m_dn = pair ? 256 : 128;

    FfnArgs a;
    memset(&a, 0, sizeof a);
    for (int pi = 0; pi < n_probs; ++pi) {
        const FfnProblem &P = probs[pi];
        const int I = I_pp[pi];
        if (fp8) {
            const long long pitch = fp8_scale_pitch(P.rows);
            if (!encode_weight8(&a.upA[pi], P.W1, P.n_groups, I, H) ||
                !encode_weight8(&a.upA3[pi], P.W3, P.n_groups, I, H) ||
                !encode_act8(&a.upB[pi], P.act, P.rows, H, bn) ||
                !encode_scales(&a.upS[pi], P.act_s, P.rows, pitch, H / 128, bn + 4) ||
                !encode_weight8(&a.dnA[pi], P.W2, P.n_groups, H, I) ||
                !encode_act8(&a.dnB[pi], P.h8, P.rows, I, bn) ||
                !encode_scales(&a.dnS[pi], P.h_s, P.rows, pitch, I / 128, bn + 4))
                return cudaErrorInvalidValue;
        } else if (!encode_weight(&a.upA[pi], P.W1, P.n_groups, H, I) ||
                   !encode_weight(&a.upA3[pi], P.W3, P.n_groups, H, I) ||
                   !encode_act(&a.upB[pi], P.act, P.rows, H, bn_cta) ||
                   !encode_weight(&a.dnA[pi], P.W2, P.n_groups, I, H) ||
                   !encode_act(&a.dnB[pi], P.h, P.rows, I, bn_cta)) {
            return cudaErrorInvalidValue;
        }
        ProbDev d{};
        d.offsets = P.offsets;
        d.n_groups = P.n_groups;
        d.dense_rows = P.dense_rows;
        d.rows = P.rows;
        // FP8 tiles: 128 columns of I (up), 256 rows of H (down)
        d.mt_up = fp8 ? (I + 127) / 128 : (I + m_up - 1) / m_up;
        d.mt_dn = fp8 ? (H + 255) / 256 : (H + m_dn - 1) / m_dn;
        d.kb_up = H / (fp8 ? BK8 : BK);
        d.kb_dn = I / (fp8 ? BK8 : BK);
        d.I = I;
        d.H = H;
        d.out_fp32 = P.out_fp32;
        d.h = P.h;
        d.out = P.out;
        d.s1 = P.S1;
        d.s3 = P.S3;
        d.s2 = P.S2;
        a.prob[pi] = d;
    }
    a.n_probs = n_probs;
    a.bn = bn;
    a.stages = stages;
    a.tmem_cols = tcols;
    a.tab = tab;
    a.ready = ready;
    a.status = status;
    a.timeout_ns = timeout_ns;
    a.inject = inject;
    a.phase_only = phase_only;
    const size_t slots = ffn_ready_slots(rows_total, n_cg);
    cudaError_t err;
    if (!ready_zeroed && (err = cudaMemsetAsync(ready, 0, slots * sizeof(unsigned), s)) != cudaSuccess)
        return err;
    const void *fn = fp8 ? reinterpret_cast<const void *>(ffn_kernel<false, true>)
                         : (pair ? reinterpret_cast<const void *>(ffn_kernel<true, false>)
                                 : reinterpret_cast<const void *>(ffn_kernel<false, false>));
    if ((err = ensure_smem(fn, smem)) != cudaSuccess) return err;
    // the tile counters of a launch: the last readiness slot, the one before it for a
    // launch of the down tiles alone (the up tiles' launch ran first with the last slot)
    a.next_tile = ready + slots - (phase_only == 1 ? 2 : 1);
    const dim3 block(fp8 ? NUM_THREADS_FP8 : NUM_THREADS);
    const int n_cta = max_ctas > 0 && max_ctas < num_sms() ? max_ctas : num_sms();
    const dim3 grid_pair(n_cta / 2 > 0 ? n_cta / 2 * 2 : 2), grid_one(n_cta);
    if (fp8)
        err = launch_pdl(ffn_kernel<false, true>, grid_one, block, smem, s, 1, a);
    else
        err = pair ? launch_pdl(ffn_kernel<true, false>, grid_pair, block, smem, s, 2, a)
                   : launch_pdl(ffn_kernel<false, false>, grid_one, block, smem, s, 1, a);
    if (err != cudaSuccess) return err;
    // one launch computes both projections: the "between" mark follows it
    if (mid_event && (err = cudaEventRecord(mid_event, s)) != cudaSuccess) return err;
    return cudaSuccess;
}

}  // namespace moe
