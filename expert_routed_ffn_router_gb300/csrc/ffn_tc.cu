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
// FP8 weights (ffn_kernel<PAIR, true>).  The weights arrive as E4M3 bytes with one
// power-of-two scale per 128 x 128 tile ("Lower latency and higher throughput...",
// Quantization).  The ring then holds token rows and E4M3 weight boxes; eight more warps
// dequantise each box into the bf16 tile the MMA reads (exact: q * 2^k fits bf16) in a
// separate small ring of tiles.  The MMAs and the epilogue are those of the bf16 kernel.
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
constexpr int CONV_WARPS = 8;             // warps that dequantise the FP8 weight tiles
constexpr int NUM_THREADS_FP8 = NUM_THREADS + 32 * CONV_WARPS;
constexpr int A8_BYTES = BM * BK;          // 8 KB: the stage's weight tile as E4M3 bytes
constexpr int FP8_END = 1 << 20;          // scale slot value that tells the converters to stop
constexpr int FP8_SB = 3;                 // FP8: slots of dequantised weight tiles
constexpr int TSC = 128;                  // FP8: scale-table entries per box (H, I <= 16384)
constexpr int MAX_STAGES_FP8 = 24;        // FP8: the E4M3 ring is deeper (its stages are small)
constexpr int MAX_GROUPS = 1024;          // groups of one problem
constexpr int MAX_CG = 1040;              // groups of all problems of a launch
constexpr int CW = 32;                    // epilogue chunk: accumulator columns per TMEM load
constexpr int XCHG_FLOATS = 2 * CW * 64;  // double-buffered G exchange (up epilogue)
constexpr int PH_UP = 0, PH_DOWN = 1;
constexpr int TQ = 4;                     // depth of the ring that hands claimed tiles to the roles
constexpr int NT_BLOCK = 8;               // token tiles per block of a group's tile order
constexpr int MAX_STAGES = 8;       // deeper rings measured slower at decode (HBM-bound up projection)

struct ProbDev {
    const int32_t *offsets;  // [n_groups + 1] on the device, or nullptr (one dense group)
    int n_groups;
    int dense_rows;
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

// generic-proxy shared-memory stores -> later async-proxy (tensor core) reads
__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <bool PAIR, bool FP8>
__global__ void __launch_bounds__(FP8 ? NUM_THREADS_FP8 : NUM_THREADS, 1)
    ffn_kernel(const __grid_constant__ FfnArgs p)
{
    constexpr int NT = FP8 ? NUM_THREADS_FP8 : NUM_THREADS;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int bn = p.bn, S = p.stages, tab = p.tab;
    const int bn_cta = PAIR ? bn / 2 : bn;    // token rows of B staged in this CTA
    // stage: weight tile (bf16, SW128) | token rows.  With FP8 weights the ring's stages hold
    // token rows | E4M3 weight bytes, and the dequantised weight tiles have a ring of their
    // own (FP8_SB slots), so the E4M3 ring can be deep enough to keep HBM busy
    const int stage_bytes = FP8 ? bn_cta * 128 + A8_BYTES : A_BYTES + bn_cta * 128;
    const int b_off = FP8 ? 0 : A_BYTES;                      // token rows within a stage
    unsigned char *stage_base = smem;
    unsigned char *abf_base = smem + static_cast<size_t>(S) * stage_bytes;   // FP8 only
    float *xbuf = reinterpret_cast<float *>(abf_base + (FP8 ? FP8_SB * A_BYTES : 0));
    uint64_t *full = reinterpret_cast<uint64_t *>(xbuf + XCHG_FLOATS);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *tqf = drain + 1;                                // [TQ] tile slot written
    uint64_t *tqe = tqf + TQ;                                 // [TQ] tile slot read by all roles
    uint64_t *cvt = tqe + TQ;                                 // [FP8_SB] FP8: slot dequantised
    uint64_t *cempty = cvt + (FP8 ? FP8_SB : 0);              // [FP8_SB] FP8: slot consumed
    int *sc8 = reinterpret_cast<int *>(cempty + (FP8 ? FP8_SB : 0));   // [S][2] box scale exponents
    int *tsc = sc8 + (FP8 ? 2 * S : 0);                       // [2][TSC] FP8: the tile's scales
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tsc + (FP8 ? 2 * TSC : 0));
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
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], PAIR ? 256 : 128);
        }
        mbar_init(drain, 1);
        for (int q = 0; q < TQ; ++q) {
            mbar_init(&tqf[q], 1);
            // consumers of a slot: MMA and epilogue (and in a pair the odd CTA's producer
            // and epilogue, which read their copy of the slot)
            mbar_init(&tqe[q], PAIR ? 4 : 2);
        }
        if (FP8)
            for (int q = 0; q < FP8_SB; ++q) {
                mbar_init(&cvt[q], PAIR ? 2 * CONV_WARPS : CONV_WARPS);
                mbar_init(&cempty[q], 1);
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
    for (int pi = 0; pi < p.n_probs; ++pi) {
        const ProbDev &P = p.prob[pi];
        const int base = pi ? n0 : 0;
        for (int g = tid; g < P.n_groups; g += NT) {
            const int a = P.offsets ? P.offsets[g] : 0;
            const int b = P.offsets ? P.offsets[g + 1] : P.dense_rows;
            gstart[base + g] = a;
            gm[base + g] = b - a;
        }
    }
    __syncthreads();
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
    auto tqe_arrive = [&](int q) {
        if (PAIR) mbar_arrive_cluster(mapa_shared(smem_u32(&tqe[q]), 0));
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
            auto claim = [&](Tile &T) -> bool {
                if (!mbar_wait(&tqe[qs], qph ^ 1u, abort_flag, p.status, tmo)) return false;
                const int t = t_begin + static_cast<int>(atomicAdd(p.next_tile, 1u));
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
                    // CTA pairs claim the following tile before this tile's loads are issued,
                    // so the global atomic, the decode and the hand-over to the odd CTA
                    // overlap them instead of stalling the ring at the tile boundary (single-
                    // CTA decode tiles measured better claiming one tile at a time)
                    if (PAIR && T.ph >= 0) {
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
                const int brow = T.row0 + (PAIR && !leader ? n_mma_of(T) / 2 : 0);
                const int kblocks = up ? P.kb_up : P.kb_dn;
                // FP8: scale exponents of the two weight boxes of stage kb (a box past the
                // last weight column reads zeros: any tile's scale does, so its index is
                // clamped to the last tile of the row)
                // The tile's scales (one per 128 K rows and box) are copied into a shared
                // table when the tile starts (asynchronous 4-byte copies, all in flight
                // together), so the per-stage loop reads them from shared memory.
                if (FP8) {
                    const int nkq = (kblocks * BK + 127) / 128;
                    const int nc = (up ? P.I : P.H) / 128;
                    const int nr = (up ? P.H : P.I) / 128;
                    for (int box = 0; box < 2; ++box) {
                        const int c = min((box ? a1 : a0) / 128, nc - 1);
                        const int32_t *src = (up ? (box ? P.s3 : P.s1) : P.s2) +
                                             static_cast<size_t>(T.g) * nr * nc + c;
                        for (int q = 0; q < nkq; ++q)
                            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;"
                                         ::"r"(smem_u32(tsc + box * TSC + q)),
                                           "l"(reinterpret_cast<uint64_t>(src + static_cast<size_t>(q) * nc))
                                         : "memory");
                    }
                    asm volatile("cp.async.commit_group;" ::: "memory");
                    asm volatile("cp.async.wait_group 0;" ::: "memory");
                }
                if (!up) {
                    // the h rows of this token tile are complete once every up-projection
                    // weight tile of it has been stored (each CTA of a pair stores half)
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
                        // E4M3 weight boxes into the stage's byte area, token rows as usual;
                        // each CTA's copies complete on its own barrier, where its converter
                        // warps wait (they then tell the MMA issuer)
                        sc8[2 * s] = tsc[(kb * BK) / 128];
                        sc8[2 * s + 1] = tsc[TSC + (kb * BK) / 128];
                        unsigned char *a8 = a + bn_cta * 128;
                        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(A8_BYTES + bn_cta * 128));
                        tma_load_3d(a8, mA, &full[s], a0, kb * BK, T.g);
                        tma_load_3d(a8 + A8_BYTES / 2, mA2, &full[s], a1, kb * BK, T.g);
                        tma_load_2d(a, mB, &full[s], kb * BK, brow);
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
            if (FP8 && ok) {
                // the converter warps stop at a stage whose scale slot says so (after the
                // drain above: this arrival moves the stage's barrier one phase on)
                if (mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status, tmo)) {
                    sc8[2 * s] = FP8_END;
                    mbar_arrive(&full[s]);
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
            const uint64_t adesc0 = smem_desc_sw128(FP8 ? smem_u32(abf_base) : ring0, HALF_A, 1024);
            const uint64_t bdesc0 = smem_desc_sw128(ring0 + b_off, 16, 1024);
            const uint32_t stage16 = static_cast<uint32_t>(stage_bytes) >> 4;  // descriptor units
            uint32_t s = 0, ph = 0, soff = 0, tc = 0;
            uint32_t sb = 0, pb = 0, aoff = 0;          // FP8: slot of the dequantised tile
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
                if (!mbar_wait(&tempty[b], tph ^ 1u, abort_flag, p.status, tmo)) { ok = false; break; }
                tc_fence_after();
                const int n_mma = n_mma_of(T);
                const uint32_t idesc = idesc_bf16_f32(PAIR ? 2 * BM : BM, static_cast<uint32_t>(n_mma), true, false);
                const uint32_t d_tmem = tmem_base + b * static_cast<uint32_t>(bn);
                const int kblocks = T.ph == PH_UP ? P.kb_up : P.kb_dn;
                for (int kb = 0; kb < kblocks; ++kb) {
                    // FP8: the stage is ready once every converter warp (of both CTAs of a
                    // pair) has written its dequantised weight tile (after the stage's copies)
                    const bool got = !FP8 ? mbar_wait(&full[s], ph, abort_flag, p.status, tmo)
                                     : PAIR ? mbar_wait_cluster(&cvt[sb], pb, abort_flag, p.status, tmo)
                                            : mbar_wait(&cvt[sb], pb, abort_flag, p.status, tmo);
                    if (!got) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = adesc0 + (FP8 ? aoff : soff), bd = bdesc0 + soff;
                    // K16 steps: +2048 B along A (MN-major), +32 B along B (K-major)
                    if (PAIR) {
                        tc_mma_bf16_pair(d_tmem, ad, bd, idesc, kb != 0 ? 1u : 0u);
                        tc_mma_bf16_pair(d_tmem, ad + 128, bd + 2, idesc, 1u);
                        tc_mma_bf16_pair(d_tmem, ad + 256, bd + 4, idesc, 1u);
                        tc_mma_bf16_pair(d_tmem, ad + 384, bd + 6, idesc, 1u);
                        tc_commit_pair_mc(&empty[s], 3);
                        if (FP8) tc_commit_pair_mc(&cempty[sb], 3);
                    } else {
                        tc_mma_bf16(d_tmem, ad, bd, idesc, kb != 0 ? 1u : 0u);
                        tc_mma_bf16(d_tmem, ad + 128, bd + 2, idesc, 1u);
                        tc_mma_bf16(d_tmem, ad + 256, bd + 4, idesc, 1u);
                        tc_mma_bf16(d_tmem, ad + 384, bd + 6, idesc, 1u);
                        tc_commit(&empty[s]);
                        if (FP8) tc_commit(&cempty[sb]);
                    }
                    if (++s == static_cast<uint32_t>(S)) { s = 0; ph ^= 1u; soff = 0; } else { soff += stage16; }
                    if (FP8) {
                        if (++sb == static_cast<uint32_t>(FP8_SB)) { sb = 0; pb ^= 1u; aoff = 0; }
                        else { aoff += static_cast<uint32_t>(A_BYTES) >> 4; }
                    }
                }
                if (!ok) break;
                if (PAIR) tc_commit_pair_mc(&tfull[b], 3); else tc_commit(&tfull[b]);
            }
            // drain: every MMA issued by this thread has completed before TMEM is freed
            if (PAIR) tc_commit_pair_mc(drain, 1); else tc_commit(drain);
            int dummy_abort = 0;
            mbar_wait(drain, 0, &dummy_abort, nullptr, 20000000ull);
        }
    } else if (FP8 && warp >= 6) {
        // ------------------------------------------------------- FP8 weight converters
        // Each stage's two E4M3 boxes (64 K rows x 64 weight columns, 64-byte rows) become
        // the bf16 weight tile in the swizzled layout TMA gives bf16 boxes (128-byte rows,
        // 16-byte chunk c of row r at chunk c ^ (r & 7)), times the box's scale 2^k (exact).
        // 16-byte chunks of E4M3 spread over the converter threads; then a proxy fence so
        // the tensor core sees the generic stores, and one arrival per warp.
        const int ct = tid - NUM_THREADS;
        const uint32_t cvt_c0 = PAIR ? mapa_shared(smem_u32(cvt), 0) : 0u;   // even CTA's cvt[0]
        uint32_t s = 0, ph = 0, sb = 0, pb = 0;
        for (;;) {
            if (!mbar_wait(&full[s], ph, abort_flag, p.status, tmo)) break;
            const int k0 = sc8[2 * s], k1 = sc8[2 * s + 1];
            if (k0 == FP8_END) break;
            if (!mbar_wait(&cempty[sb], pb ^ 1u, abort_flag, p.status, tmo)) break;
            const uint32_t abf = smem_u32(abf_base) + sb * static_cast<uint32_t>(A_BYTES);
            const uint32_t a8 = smem_u32(stage_base) + s * static_cast<uint32_t>(stage_bytes) +
                                static_cast<uint32_t>(bn_cta) * 128u;
            // every chunk's bytes first (independent shared loads), then the conversions
            constexpr int NCH = 16 / CONV_WARPS;
            uint32_t w[NCH][4];
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
                const uint32_t addr = a8 + 16u * static_cast<uint32_t>(ct + 32 * CONV_WARPS * j);
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(w[j][0]), "=r"(w[j][1]), "=r"(w[j][2]), "=r"(w[j][3]) : "r"(addr));
            }
            // bit moves (x 2^-120) then one packed multiply by 2^(120 + k): a power of two,
            // so exact, and the results are normal bf16 for -117 <= k <= 7; other scales go
            // through fp32 (exact power-of-two products)
            const bool fast = k0 >= -117 && k0 <= 7 && k1 >= -117 && k1 <= 7;
            const uint32_t e0 = static_cast<uint32_t>(247 + k0) << 7, e1 = static_cast<uint32_t>(247 + k1) << 7;
            const uint32_t sc_a = e0 | (e0 << 16), sc_b = e1 | (e1 << 16);
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
                const int chunk = ct + 32 * CONV_WARPS * j;   // 0..511 over the two 4 KB boxes
                const int box = chunk >> 8, r = (chunk >> 2) & 63, cq = chunk & 3;
                uint32_t o[8];
                if (fast) {
                    const uint32_t sc2 = box ? sc_b : sc_a;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t x, y;
                        e4m3x4_to_bf16x2_shifted(w[j][i], x, y);
                        o[2 * i] = bf16x2_mul(x, sc2);
                        o[2 * i + 1] = bf16x2_mul(y, sc2);
                    }
                } else {
                    const float sc = pow2f(box ? k1 : k0);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f0 = e4m3x2_to_f32x2(static_cast<uint16_t>(w[j][i] & 0xffffu));
                        const float2 f1 = e4m3x2_to_f32x2(static_cast<uint16_t>(w[j][i] >> 16));
                        o[2 * i] = f32x2_to_bf16x2(f0.y * sc, f0.x * sc);
                        o[2 * i + 1] = f32x2_to_bf16x2(f1.y * sc, f1.x * sc);
                    }
                }
                const uint32_t row = abf + static_cast<uint32_t>(box * HALF_A + r * 128);
                const uint32_t d0 = row + ((static_cast<uint32_t>(2 * cq) ^ static_cast<uint32_t>(r & 7)) << 4);
                const uint32_t d1 = row + ((static_cast<uint32_t>(2 * cq + 1) ^ static_cast<uint32_t>(r & 7)) << 4);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                             ::"r"(d0), "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]) : "memory");
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                             ::"r"(d1), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7]) : "memory");
            }
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
                if (PAIR) mbar_arrive_cluster(cvt_c0 + 8u * sb);
                else mbar_arrive(&cvt[sb]);
            }
            if (++s == static_cast<uint32_t>(S)) { s = 0; ph ^= 1u; }
            if (++sb == static_cast<uint32_t>(FP8_SB)) { sb = 0; pb ^= 1u; }
        }
    } else {
        // ----------------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        uint32_t tc = 0, cc = 0;
        uint32_t qs = 0, qph = 0;
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
            const bool ok = mbar_wait(&tfull[b], tph, abort_flag, p.status, tmo);
            if (!epi_all(ok)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * static_cast<uint32_t>(bn);
            const int nchunks = (T.nvalid + CW - 1) / CW;
            const int mt = mt_cta(T);
            // one chunk = CW token columns of this warp's 32 accumulator rows (a 16-row
            // tile has only 16 columns per buffer)
            auto load_chunk = [&](int c, float (&v)[CW]) {
                __syncwarp();
                if (bn >= CW) {
                    tmem_ld32(tbase + CW * c, v);
                } else {
                    float h[16];
                    tmem_ld16(tbase, h);
#pragma unroll
                    for (int j = 0; j < 16; ++j) { v[j] = h[j]; v[j + 16] = 0.f; }
                }
            };
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
                // stores, read later by other SMs' TMA)
                fence_proxy_async_global();
                __threadfence();
                named_bar_sync(3, 128);
                if (warp == 2 && lane == 0) atomicAdd(p.ready + T.nti, 1u);
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
            tc_fence_before();
            if (PAIR)
                mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[b]), 0));
            else
                mbar_arrive(&tempty[b]);
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

// 3-D weight tensor [n_groups][rows][cols] (cols contiguous), 64 x 64 boxes: bf16 into the
// 128-byte swizzle the MMA reads, or E4M3 bytes (fp8) as plain 64-byte rows.
bool encode_weight(CUtensorMap *m, const void *base, int n_groups, int rows, int cols,
                   bool fp8 = false)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t esz = fp8 ? 1 : 2;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(n_groups)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * esz,
                             static_cast<cuuint64_t>(cols) * rows * esz};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
    const size_t stage = fp8 ? static_cast<size_t>(bn_cta) * 128 + A8_BYTES
                             : static_cast<size_t>(A_BYTES) + bn_cta * 128;
    return 1024 + stages * stage + (fp8 ? static_cast<size_t>(FP8_SB) * A_BYTES : 0) +
           XCHG_FLOATS * 4 + (2 * stages + 5 + 2 * TQ) * 8 + (fp8 ? 2 * FP8_SB * 8 + stages * 8 + 2 * TSC * 4 : 0) +
           16 + (6 * static_cast<size_t>(tab) + 8 * TQ) * 4;
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
        if (fp8 && (!probs[pi].S1 || !probs[pi].S3 || !probs[pi].S2 || H % 128 || I_pp[pi] % 128 ||
                    H > 128 * TSC || I_pp[pi] > 128 * TSC))
            return cudaErrorInvalidValue;
        n_cg += probs[pi].n_groups;
        rows_total += probs[pi].rows;
    }
    if (n_cg > MAX_CG) return cudaErrorInvalidValue;
    int bn = pick_bn(token_hint);
    bool pair = g_variant == 2 || (g_variant == 0 && bn >= PAIR_MIN_BN);
    if (pair && bn < 32) bn = 32;           // 16 token rows per CTA at least
    const int bn_cta = pair ? bn / 2 : bn;
    const int tab = (n_cg + 1 + 3) & ~3;
    const int stages = pick_stages(bn_cta, tab, fp8);
    const size_t smem = ffn_smem_bytes(bn_cta, stages, tab, fp8);
    int tcols = 32;
    while (tcols < 2 * bn) tcols <<= 1;
    const int m_up = pair ? 128 : 64;      // weight columns of one tile
    const int m_dn = pair ? 256 : 128;

    FfnArgs a;
    memset(&a, 0, sizeof a);
    for (int pi = 0; pi < n_probs; ++pi) {
        const FfnProblem &P = probs[pi];
        const int I = I_pp[pi];
        if (!encode_weight(&a.upA[pi], P.W1, P.n_groups, H, I, fp8) ||
            !encode_weight(&a.upA3[pi], P.W3, P.n_groups, H, I, fp8) ||
            !encode_act(&a.upB[pi], P.act, P.rows, H, bn_cta) ||
            !encode_weight(&a.dnA[pi], P.W2, P.n_groups, I, H, fp8) ||
            !encode_act(&a.dnB[pi], P.h, P.rows, I, bn_cta))
            return cudaErrorInvalidValue;
        ProbDev d{};
        d.offsets = P.offsets;
        d.n_groups = P.n_groups;
        d.dense_rows = P.dense_rows;
        d.mt_up = (I + m_up - 1) / m_up;
        d.mt_dn = (H + m_dn - 1) / m_dn;
        d.kb_up = H / 64;
        d.kb_dn = I / 64;
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
    const void *fn = fp8 ? (pair ? reinterpret_cast<const void *>(ffn_kernel<true, true>)
                                 : reinterpret_cast<const void *>(ffn_kernel<false, true>))
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
        err = pair ? launch_pdl(ffn_kernel<true, true>, grid_pair, block, smem, s, 2, a)
                   : launch_pdl(ffn_kernel<false, true>, grid_one, block, smem, s, 1, a);
    else
        err = pair ? launch_pdl(ffn_kernel<true, false>, grid_pair, block, smem, s, 2, a)
                   : launch_pdl(ffn_kernel<false, false>, grid_one, block, smem, s, 1, a);
    if (err != cudaSuccess) return err;
    // one launch computes both projections: the "between" mark follows it
    if (mid_event && (err = cudaEventRecord(mid_event, s)) != cudaSuccess) return err;
    return cudaSuccess;
}

}  // namespace moe
