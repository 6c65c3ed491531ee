// dispatch.cu -- the single-GPU counterpart of the AllToAll Dispatch: per-expert counts,
// exclusive scan, a deterministic stable permutation of the (token, slot) pairs into
// expert-contiguous rows, the row gather, and the expert co-activation (affinity) matrix.
//
// Method: "Lower latency and higher throughput with multi-node DeepSeek deployment",
// section "Expert Parallelism" (tokens are sent to the GPUs of their experts before the
// expert computation) and section "MoE Router" (a dense dispatch/combine needs routing
// information aggregated per expert, not per token).  The affinity matrix is the expert
// co-activation matrix A of "GRACE-MoE", Core Idea 1 (Expert Grouping).
//
// Representation: the 0/1 selection matrix S[T, E] is stored as 32-token bit masks,
// smask[w][e] = bit l set iff token 32w + l chose expert e.  Every quantity is a popcount of
// these words, so nothing depends on the order in which atomics land:
//   counts[e]         = sum_w popc(smask[w][e])
//   rank of token t   = #{t' < t : t' chose e}  (prefix popcount -> stable order)
//   affinity[i][j]    = sum_w popc(smask[w][i] & smask[w][j]),  i != j
// The masks of a warp are built with warp-aggregated shared-memory atomics
// (__match_any_sync groups the lanes that picked the same expert).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int CHUNK = 256;            // tokens per chunk (8 warps x 32)
constexpr int CW = CHUNK / 32;        // mask rows per chunk
constexpr int KMAX = 32;              // largest top-K

// The K (<= 32) expert indices of token t, all loads issued before any is used (-1 for an
// invalid token); one memory round trip instead of K.
__device__ __forceinline__ void load_topk(const int32_t *__restrict__ idx, int t, bool valid,
                                          int K, int (&ev)[KMAX])
{
#pragma unroll
    for (int j = 0; j < KMAX; ++j) ev[j] = (valid && j < K) ? idx[static_cast<size_t>(t) * K + j] : -1;
}

__global__ void __launch_bounds__(CHUNK) masks_kernel(const int32_t *__restrict__ idx, int T,
                                                      int E, int K, uint32_t *smask,
                                                      int32_t *chunk_cnt, int *status)
{
    pdl_wait();
    extern __shared__ uint32_t m_s[];    // [CW][E]
    const int c = blockIdx.x, tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31;
    for (int i = tid; i < CW * E; i += CHUNK) m_s[i] = 0u;
    __syncthreads();
    const int t = c * CHUNK + tid;
    const bool valid = t < T;
    int ev[KMAX];
    load_topk(idx, t, valid, K, ev);
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        if (j >= K) break;
        int e = ev[j];
        if (valid && (e < 0 || e >= E)) {
            report(status, MOE_ERR_INVALID_ARG);
            e = -1;
        }
        const uint32_t peers = __match_any_sync(kFullMask, e);
        if (e >= 0 && lane == __ffs(peers) - 1) atomicOr(&m_s[w * E + e], peers);
    }
    __syncthreads();
    const int rows = min(CW, (T - c * CHUNK + 31) / 32);
    for (int i = tid; i < rows * E; i += CHUNK)
        smask[static_cast<size_t>(c * CW) * E + i] = m_s[i];
    for (int e = tid; e < E; e += CHUNK) {
        int n = 0;
        for (int r = 0; r < CW; ++r) n += __popc(m_s[r * E + e]);
        chunk_cnt[static_cast<size_t>(c) * E + e] = n;
    }
}

// One CTA: per-expert totals, exclusive scan over experts, per-chunk bases.
__global__ void __launch_bounds__(1024) scan_kernel(int E, int n_chunks,
                                                    const int32_t *chunk_cnt,
                                                    int32_t *chunk_base, int32_t *counts,
                                                    int32_t *offsets)
{
    pdl_wait();
    __shared__ int warp_sums[32];
    const int e = threadIdx.x, lane = e & 31, w = e >> 5;
    int total = 0;
    if (e < E)
        for (int c = 0; c < n_chunks; ++c) {
            const int n = chunk_cnt[static_cast<size_t>(c) * E + e];
            chunk_base[static_cast<size_t>(c) * E + e] = total;
            total += n;
        }
    // block-wide exclusive scan of `total` over experts
    int incl = total;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(kFullMask, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
        int v = lane < blockDim.x / 32 ? warp_sums[lane] : 0;
        int inc = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(kFullMask, inc, off);
            if (lane >= off) inc += u;
        }
        warp_sums[lane] = inc - v;
    }
    __syncthreads();
    const int excl = warp_sums[w] + incl - total;
    if (e < E) {
        counts[e] = total;
        offsets[e] = excl;
        for (int c = 0; c < n_chunks; ++c) chunk_base[static_cast<size_t>(c) * E + e] += excl;
    }
    if (e == E - 1) offsets[E] = excl + total;
}

__global__ void __launch_bounds__(CHUNK) scatter_kernel(const int32_t *__restrict__ idx, int T,
                                                        int E, int K, const uint32_t *smask,
                                                        const int32_t *chunk_base, int32_t *perm,
                                                        int32_t *slot_pos)
{
    pdl_wait();
    extern __shared__ uint32_t sh[];
    uint32_t *m_s = sh;                                  // [CW][E]
    int32_t *base = reinterpret_cast<int32_t *>(sh + CW * E);  // [CW][E]
    const int c = blockIdx.x, tid = threadIdx.x;
    const int w = tid >> 5, lane = tid & 31;
    const int rows = min(CW, (T - c * CHUNK + 31) / 32);
    for (int i = tid; i < CW * E; i += CHUNK)
        m_s[i] = i < rows * E ? smask[static_cast<size_t>(c * CW) * E + i] : 0u;
    __syncthreads();
    for (int e = tid; e < E; e += CHUNK) {
        int run = chunk_base[static_cast<size_t>(c) * E + e];
        for (int r = 0; r < CW; ++r) {
            base[r * E + e] = run;
            run += __popc(m_s[r * E + e]);
        }
    }
    __syncthreads();
    const int t = c * CHUNK + tid;
    if (t >= T) return;
    const uint32_t below = (1u << lane) - 1u;
    int ev[KMAX];
    load_topk(idx, t, true, K, ev);
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        if (j >= K) break;
        const int e = ev[j];
        if (e < 0 || e >= E) {           // reported by masks_kernel; no row for this pair
            slot_pos[static_cast<size_t>(t) * K + j] = -1;
            continue;
        }
        const int r = base[w * E + e] + __popc(m_s[w * E + e] & below);
        slot_pos[static_cast<size_t>(t) * K + j] = r;
        perm[r] = t;
    }
}

// Xp[r] = X[perm[r]] for r < offsets[E]; one warp per row, 16-byte vectors (X small enough
// to stay in L2: many rows in flight).  `gb` / `ngb` are this block's index and the block
// count of the gather part of the launch.
__device__ __forceinline__ void gather_rows(const uint4 *__restrict__ X, int H,
                                            const int32_t *__restrict__ perm,
                                            const int32_t *__restrict__ offsets, int E,
                                            uint4 *__restrict__ Xp, int gb, int ngb)
{
    const int n_rows = offsets[E];
    const int vec = H / 8;
    const int lane = threadIdx.x & 31;
    const int gw = (gb * blockDim.x + threadIdx.x) >> 5;
    const int nw = (ngb * blockDim.x) >> 5;
    for (int r = gw; r < n_rows; r += nw) {
        const uint4 *src = X + static_cast<size_t>(perm[r]) * vec;
        uint4 *dst = Xp + static_cast<size_t>(r) * vec;
        int v = lane;
        for (; v + 96 < vec; v += 128) {
            const uint4 a0 = __ldg(src + v), a1 = __ldg(src + v + 32);
            const uint4 a2 = __ldg(src + v + 64), a3 = __ldg(src + v + 96);
            dst[v] = a0; dst[v + 32] = a1; dst[v + 64] = a2; dst[v + 96] = a3;
        }
        for (; v < vec; v += 32) dst[v] = __ldg(src + v);
    }
}

// Xp[slot_pos[t][j]] = X[t] for every token t and slot j < K, token by token: one warp per
// token reads its row once (16-byte vectors, 2 KB in flight per warp) and writes it to its K
// destination rows.  Used when X is larger than about half of L2: gathering row by row in
// Xp order then re-reads each token row K times from HBM.
__device__ __forceinline__ void gather_tokens(const uint4 *__restrict__ X, int T, int H, int K,
                                            const int32_t *__restrict__ slot_pos,
                                            uint4 *__restrict__ Xp, int gb, int ngb)
{
    const int vec = H / 8;
    const int lane = threadIdx.x & 31;
    const int gw = (gb * blockDim.x + threadIdx.x) >> 5;
    const int nw = (ngb * blockDim.x) >> 5;
    for (int t = gw; t < T; t += nw) {
        const uint4 *src = X + static_cast<size_t>(t) * vec;
        int dst_row = 0;
        if (lane < K) dst_row = slot_pos[static_cast<size_t>(t) * K + lane];
        for (int v0 = 0; v0 < vec; v0 += 128) {
            uint4 a[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + 32 * u + lane;
                a[u] = v < vec ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
            }
            for (int j = 0; j < K; ++j) {
                const int row = __shfl_sync(kFullMask, dst_row, j);
                if (row < 0) continue;   // a pair with an out-of-range expert: no row
                uint4 *dst = Xp + static_cast<size_t>(row) * vec;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int v = v0 + 32 * u + lane;
                    if (v < vec) dst[v] = a[u];
                }
            }
        }
    }
}

// affinity[i][j] = sum_w popc(smask[w][i] & smask[w][j]) for i != j, 0 on the diagonal.
__device__ __forceinline__ void affinity_tile(const uint32_t *__restrict__ smask, int n_words,
                                              int E, int32_t *aff, int bi, int bj)
{
    __shared__ uint32_t A[64][33];
    __shared__ uint32_t B[64][33];
    const int i0 = bi * 32, j0 = bj * 32;
    const int tid = threadIdx.x;
    const int ti = tid >> 3, tj = (tid & 7) * 4;
    int acc[4] = {0, 0, 0, 0};
    for (int w0 = 0; w0 < n_words; w0 += 64) {
        for (int q = tid; q < 64 * 32; q += 256) {
            const int r = q >> 5, col = q & 31;
            const int w = w0 + r;
            const bool ok = w < n_words;
            A[r][col] = (ok && i0 + col < E) ? smask[static_cast<size_t>(w) * E + i0 + col] : 0u;
            B[r][col] = (ok && j0 + col < E) ? smask[static_cast<size_t>(w) * E + j0 + col] : 0u;
        }
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < 64; ++r) {
            const uint32_t a = A[r][ti];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] += __popc(a & B[r][tj + q]);
        }
        __syncthreads();
    }
    const int i = i0 + ti;
    if (i >= E) return;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int j = j0 + tj + q;
        if (j < E) aff[static_cast<size_t>(i) * E + j] = (i == j) ? 0 : acc[q];
    }
}

// The data-parallel tail of dispatch in one launch (no dependency between its parts): the
// first n_aff blocks compute 32x32 tiles of the affinity matrix, the others gather the
// permuted rows and zero `zero_n` words of `zero_buf` (the expert FFN's readiness
// counters, so that its launch needs no separate memset).
__global__ void __launch_bounds__(256) tail_kernel(const uint32_t *__restrict__ smask, int n_words,
                                                   int E, int32_t *aff, int n_aff_x, int n_aff,
                                                   const uint4 *__restrict__ X, int T, int H, int K,
                                                   const int32_t *__restrict__ slot_pos,
                                                   const int32_t *__restrict__ perm,
                                                   const int32_t *__restrict__ offsets,
                                                   uint4 *__restrict__ Xp, int by_token,
                                                   unsigned *zero_buf, int zero_n)
{
    pdl_wait();
    const int b = static_cast<int>(blockIdx.x);
    if (b < n_aff) {
        affinity_tile(smask, n_words, E, aff, b / n_aff_x, b % n_aff_x);
        return;
    }
    const int gb = b - n_aff, ngb = static_cast<int>(gridDim.x) - n_aff;
    for (int i = gb * blockDim.x + threadIdx.x; i < zero_n; i += ngb * blockDim.x) zero_buf[i] = 0u;
    if (Xp) {
        if (by_token) gather_tokens(X, T, H, K, slot_pos, Xp, gb, ngb);
        else gather_rows(X, H, perm, offsets, E, Xp, gb, ngb);
    }
}

// Small batches (T <= 256, one chunk): masks, counts, scan and stable slots of the whole
// batch in one CTA's shared memory -- the same popcount formulation as the multi-CTA
// kernels above.  m_s [CW][E] masks, off [E + 1] exclusive offsets (off[E] = rows),
// perm_s [T K] the token of every row.  With `out` the CTA also writes counts, offsets,
// perm, slot_pos and the masks to global memory.
__device__ void small_routing(const int32_t *__restrict__ idx, int T, int E, int K, uint32_t *m_s,
                              int32_t *base, int32_t *off, int32_t *perm_s, bool out,
                              int32_t *counts, int32_t *offsets, int32_t *perm,
                              int32_t *slot_pos, uint32_t *smask, int *status)
{
    __shared__ int warp_tot[CHUNK / 32];
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    for (int i = tid; i < CW * E; i += CHUNK) m_s[i] = 0u;
    __syncthreads();
    const bool valid = tid < T;
    int ev[KMAX];
    load_topk(idx, tid, valid, K, ev);
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        if (j >= K) break;
        int e = ev[j];
        if (valid && (e < 0 || e >= E)) {
            report(status, MOE_ERR_INVALID_ARG);
            e = -1;
        }
        const uint32_t peers = __match_any_sync(kFullMask, e);
        if (e >= 0 && lane == __ffs(peers) - 1) atomicOr(&m_s[w * E + e], peers);
    }
    __syncthreads();
    const int rows = (T + 31) / 32;
    if (out)
        for (int i = tid; i < rows * E; i += CHUNK) smask[i] = m_s[i];
    // counts and an exclusive scan over experts: thread tid owns experts [tid*per, +per)
    const int per = (E + CHUNK - 1) / CHUNK;
    int local = 0;
    for (int q = 0; q < per; ++q) {
        const int e = tid * per + q;
        if (e >= E) break;
        int n = 0;
        for (int r = 0; r < CW; ++r) n += __popc(m_s[r * E + e]);
        off[e] = n;              // count for now
        local += n;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    int before = 0;
    for (int q = 0; q < w; ++q) before += warp_tot[q];
    int run = before + incl - local;
    for (int q = 0; q < per; ++q) {
        const int e = tid * per + q;
        if (e >= E) break;
        const int n = off[e];
        if (out) {
            counts[e] = n;
            offsets[e] = run;
        }
        off[e] = run;
        run += n;
    }
    if (tid == CHUNK - 1) {
        off[E] = run;
        if (out) offsets[E] = run;
    }
    __syncthreads();
    // per 32-token row bases, then the stable slot of every (token, j)
    for (int e = tid; e < E; e += CHUNK) {
        int r0 = off[e];
        for (int r = 0; r < CW; ++r) {
            base[r * E + e] = r0;
            r0 += __popc(m_s[r * E + e]);
        }
    }
    __syncthreads();
    if (valid) {
        const uint32_t below = (1u << lane) - 1u;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j >= K) break;
            const int e = ev[j];
            if (e < 0 || e >= E) {       // reported above; no row for this pair
                if (out) slot_pos[static_cast<size_t>(tid) * K + j] = -1;
                continue;
            }
            const int r = base[w * E + e] + __popc(m_s[w * E + e] & below);
            perm_s[r] = tid;
            if (out) {
                slot_pos[static_cast<size_t>(tid) * K + j] = r;
                perm[r] = tid;
            }
        }
    }
    __syncthreads();
}

// The whole dispatch of a small batch in one launch: every CTA forms the bookkeeping in its
// own shared memory (at most 256 x K entries), CTA 0 writes it out, the first n_aff CTAs
// then compute 32x32 affinity tiles from their masks and the others gather the permuted
// rows (from their own copy of perm) and zero the FFN's readiness counters.
__global__ void __launch_bounds__(CHUNK) small_dispatch_kernel(
    const int32_t *__restrict__ idx, int T, int E, int K, int32_t *counts, int32_t *offsets,
    int32_t *perm, int32_t *slot_pos, uint32_t *smask, int *status, int32_t *aff, int n_aff_x,
    int n_aff, const uint4 *__restrict__ X, int H, uint4 *__restrict__ Xp, unsigned *zero_buf,
    int zero_n)
{
    pdl_wait();
    extern __shared__ uint32_t sm[];
    uint32_t *m_s = sm;                                          // [CW][E]
    int32_t *base = reinterpret_cast<int32_t *>(sm + CW * E);    // [CW][E]
    int32_t *off = base + CW * E;                                // [E + 1]
    int32_t *perm_s = off + E + 1;                               // [T K]
    const int b = static_cast<int>(blockIdx.x);
    small_routing(idx, T, E, K, m_s, base, off, perm_s, b == 0, counts, offsets, perm, slot_pos,
                  smask, status);
    if (b < n_aff) {
        affinity_tile(m_s, (T + 31) / 32, E, aff, b / n_aff_x, b % n_aff_x);
        return;
    }
    const int gb = b - n_aff, ngb = static_cast<int>(gridDim.x) - n_aff;
    for (int i = gb * blockDim.x + threadIdx.x; i < zero_n; i += ngb * blockDim.x) zero_buf[i] = 0u;
    if (Xp) gather_rows(X, H, perm_s, off, E, Xp, gb, ngb);
}

}  // namespace

DispatchPlan dispatch_plan(int T, int E)
{
    DispatchPlan p{};
    p.n_chunks = (T + CHUNK - 1) / CHUNK;
    p.n_words = (T + 31) / 32;
    auto al = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    p.smask_bytes = al(static_cast<size_t>(p.n_chunks) * CW * E * sizeof(uint32_t));
    p.ccnt_bytes = al(static_cast<size_t>(p.n_chunks) * E * sizeof(int32_t));
    p.cbase_bytes = al(static_cast<size_t>(p.n_chunks) * E * sizeof(int32_t));
    return p;
}

cudaError_t launch_dispatch(const void *X, const int32_t *topk_idx, int T, int H, int E,
                            int K, int32_t *counts, int32_t *offsets, int32_t *perm,
                            int32_t *slot_pos, void *Xp, int32_t *affinity,
                            const DispatchPlan &plan, const DispatchScratch &scr,
                            unsigned *zero_buf, size_t zero_n, int *status, cudaStream_t s)
{
    const size_t m_smem = static_cast<size_t>(CW) * E * sizeof(uint32_t);
    cudaError_t err;
    const int n_aff_x = (E + 31) / 32;
    const int n_aff = affinity ? n_aff_x * n_aff_x : 0;
    if (T <= CHUNK) {
        // one launch: bookkeeping in every CTA, affinity tiles, row gather, counter zeroing
        long long gblocks = Xp ? (static_cast<long long>(T) * K + 7) / 8 : 1;
        const long long cap = static_cast<long long>(num_sms()) * 8;
        if (gblocks > cap) gblocks = cap;
        if (gblocks < 1) gblocks = 1;
        const size_t sm = 2 * m_smem + (E + 1 + static_cast<size_t>(T) * K) * sizeof(int32_t);
        err = ensure_smem(reinterpret_cast<const void *>(small_dispatch_kernel), sm);
        if (err != cudaSuccess) return err;
        return launch_pdl(small_dispatch_kernel, dim3(static_cast<unsigned>(n_aff + gblocks)),
                          dim3(CHUNK), sm, s, 1, topk_idx, T, E, K, counts, offsets, perm,
                          slot_pos, scr.smask, status, affinity, n_aff_x, n_aff,
                          static_cast<const uint4 *>(X), H, static_cast<uint4 *>(Xp), zero_buf,
                          static_cast<int>(zero_n));
    }
    err = ensure_smem(reinterpret_cast<const void *>(masks_kernel), m_smem);
    if (err != cudaSuccess) return err;
    err = ensure_smem(reinterpret_cast<const void *>(scatter_kernel), 2 * m_smem);
    if (err != cudaSuccess) return err;
    if ((err = launch_pdl(masks_kernel, dim3(plan.n_chunks), dim3(CHUNK), m_smem, s, 1, topk_idx, T,
                          E, K, scr.smask, scr.chunk_cnt, status)) != cudaSuccess)
        return err;
    if ((err = launch_pdl(scan_kernel, dim3(1), dim3(1024), 0, s, 1, E, plan.n_chunks,
                          static_cast<const int32_t *>(scr.chunk_cnt), scr.chunk_base, counts,
                          offsets)) != cudaSuccess)
        return err;
    if ((err = launch_pdl(scatter_kernel, dim3(plan.n_chunks), dim3(CHUNK), 2 * m_smem, s, 1,
                          topk_idx, T, E, K, static_cast<const uint32_t *>(scr.smask),
                          static_cast<const int32_t *>(scr.chunk_base), perm, slot_pos)) != cudaSuccess)
        return err;
    // affinity tiles, row gather and counter zeroing: one launch
    long long gblocks = 0;
    const bool by_token = static_cast<long long>(T) * H * 2 >= (64ll << 20);
    if (Xp) {
        gblocks = ((by_token ? static_cast<long long>(T) : static_cast<long long>(T) * K) + 7) / 8;
        const long long cap = static_cast<long long>(num_sms()) * 8;
        if (gblocks > cap) gblocks = cap;
    } else if (zero_n) {
        gblocks = 1;
    }
    if (zero_n && gblocks < 1) gblocks = 1;
    if (n_aff + gblocks == 0) return cudaSuccess;
    return launch_pdl(tail_kernel, dim3(static_cast<unsigned>(n_aff + gblocks)), dim3(256), 0, s, 1,
                      static_cast<const uint32_t *>(scr.smask), plan.n_words, E, affinity, n_aff_x,
                      n_aff, static_cast<const uint4 *>(X), T, H, K,
                      static_cast<const int32_t *>(slot_pos), static_cast<const int32_t *>(perm),
                      static_cast<const int32_t *>(offsets), static_cast<uint4 *>(Xp),
                      by_token ? 1 : 0, zero_buf, static_cast<int>(zero_n));
}

}  // namespace moe
