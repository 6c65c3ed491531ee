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
constexpr int NUM_THREADS = 192;
constexpr int MAX_GROUPS = 1024;
constexpr int XCHG_FLOATS = 2 * 16 * 64;  // double-buffered G/U exchange (up epilogue)
constexpr int MODE_UP = 0, MODE_DOWN = 1;

struct ProbDev {
    const int32_t *offsets;  // [n_groups + 1] on the device, or nullptr (one dense group)
    int n_groups;
    int dense_rows;
    int n_mtiles;            // up: I / 64; down: ceil(H / 128)
    int kblocks;             // up: H / 64; down: I / 64
    int out_ld;              // row stride of the output (elements)
    int out_cols;            // valid output columns
    int out_fp32;
    void *out;
};

struct FfnArgs {
    CUtensorMap mapA[2];     // per problem: W1 (up) or W2 (down)
    CUtensorMap mapA3[2];    // per problem: W3 (up); unused (copy of mapA) for down
    CUtensorMap mapB[2];     // per problem: activations [rows, K]
    ProbDev prob[2];
    int n_probs;
    int bn;                  // token tile: multiple of 16, <= 256
    int stages;
    int tmem_cols;
    int *status;
    unsigned long long timeout_ns;
    int inject;              // 1: the producer never fills a stage (bounded-wait test)
};

struct Tile {
    int pi, g, mt, row0, nvalid;
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

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1) ffn_kernel(const __grid_constant__ FfnArgs p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int bn = p.bn, S = p.stages;
    const int stage_bytes = A_BYTES + bn * 128;
    unsigned char *stage_base = smem;
    float *xbuf = reinterpret_cast<float *>(smem + static_cast<size_t>(S) * stage_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(xbuf + XCHG_FLOATS);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *goff = reinterpret_cast<int *>(tmem_slot + 4);       // [2][MAX_GROUPS + 1]
    int *gt = goff + 2 * (MAX_GROUPS + 1);                    // [2][MAX_GROUPS + 1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t tmo = p.timeout_ns;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int pi = 0; pi < p.n_probs; ++pi) {
            prefetch_tmap(&p.mapA[pi]);
            prefetch_tmap(&p.mapA3[pi]);
            prefetch_tmap(&p.mapB[pi]);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, static_cast<uint32_t>(p.tmem_cols));
        tmem_relinquish();
    }
    // group row offsets -> shared memory
    for (int pi = 0; pi < p.n_probs; ++pi) {
        const ProbDev &P = p.prob[pi];
        for (int g = tid; g <= P.n_groups; g += NUM_THREADS)
            goff[pi * (MAX_GROUPS + 1) + g] =
                P.offsets ? P.offsets[g] : (g == 0 ? 0 : P.dense_rows);
    }
    __syncthreads();
    // tile prefix per problem: tiles(g) = ceil(m_g / bn) * n_mtiles
    if (warp < p.n_probs) {
        const int pi = warp;
        const ProbDev &P = p.prob[pi];
        const int *go = goff + pi * (MAX_GROUPS + 1);
        int *gtp = gt + pi * (MAX_GROUPS + 1);
        int running = 0;
        for (int g0 = 0; g0 < P.n_groups; g0 += 32) {
            const int g = g0 + lane;
            int nt = 0;
            if (g < P.n_groups) {
                const int m = go[g + 1] - go[g];
                nt = m > 0 ? ((m + bn - 1) / bn) * P.n_mtiles : 0;
            }
            int incl = nt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(kFullMask, incl, off);
                if (lane >= off) incl += v;
            }
            if (g < P.n_groups) gtp[g] = running + incl - nt;
            running += __shfl_sync(kFullMask, incl, 31);
        }
        if (lane == 0) gtp[P.n_groups] = running;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_slot;
    const int total0 = gt[p.prob[0].n_groups];
    const int total = total0 + (p.n_probs > 1 ? gt[(MAX_GROUPS + 1) + p.prob[1].n_groups] : 0);

    auto decode = [&](int t) -> Tile {
        Tile T;
        T.pi = (t < total0) ? 0 : 1;
        const int lt = T.pi ? t - total0 : t;
        const ProbDev &P = p.prob[T.pi];
        const int *gtp = gt + T.pi * (MAX_GROUPS + 1);
        const int *go = goff + T.pi * (MAX_GROUPS + 1);
        int lo = 0, hi = P.n_groups;   // first index with gtp[i] > lt, minus one
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (gtp[mid] <= lt) lo = mid; else hi = mid - 1;
        }
        T.g = lo;
        const int m = go[lo + 1] - go[lo];
        const int ntn = (m + bn - 1) / bn;
        const int local = lt - gtp[lo];
        T.mt = local / ntn;
        const int nt = local - T.mt * ntn;
        T.row0 = go[lo] + nt * bn;
        T.nvalid = min(bn, m - nt * bn);
        return T;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && !p.inject) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile T = decode(t);
                const ProbDev &P = p.prob[T.pi];
                for (int kb = 0; kb < P.kblocks; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1u;
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status, tmo)) { ok = false; break; }
                    unsigned char *a = stage_base + static_cast<size_t>(s) * stage_bytes;
                    mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(stage_bytes));
                    if (MODE == MODE_UP) {
                        tma_load_3d(a, &p.mapA[T.pi], &full[s], T.mt * 64, kb * BK, T.g);
                        tma_load_3d(a + HALF_A, &p.mapA3[T.pi], &full[s], T.mt * 64, kb * BK, T.g);
                    } else {
                        tma_load_3d(a, &p.mapA[T.pi], &full[s], T.mt * 128, kb * BK, T.g);
                        tma_load_3d(a + HALF_A, &p.mapA[T.pi], &full[s], T.mt * 128 + 64, kb * BK, T.g);
                    }
                    tma_load_2d(a + A_BYTES, &p.mapB[T.pi], &full[s], kb * BK, T.row0);
                }
            }
            // every copy issued lands before the CTA can exit (a no-op wait in normal runs:
            // the MMA warp has already waited on each of these phases)
            (void)ok;
            const uint32_t n = it < static_cast<uint32_t>(S) ? it : static_cast<uint32_t>(S);
            for (uint32_t j = it - n; j < it; ++j) {
                int dummy_abort = 0;
                mbar_wait(&full[j % S], (j / S) & 1u, &dummy_abort, nullptr, 20000000ull);
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t it = 0, tc = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
                const Tile T = decode(t);
                const ProbDev &P = p.prob[T.pi];
                const uint32_t b = tc & 1u, tph = (tc >> 1) & 1u;
                if (!mbar_wait(&tempty[b], tph ^ 1u, abort_flag, p.status, tmo)) { ok = false; break; }
                tc_fence_after();
                int n_mma = (T.nvalid + 15) & ~15;
                if (n_mma > bn) n_mma = bn;
                const uint32_t idesc = idesc_bf16_f32(BM, static_cast<uint32_t>(n_mma), true, false);
                const uint32_t d_tmem = tmem_base + b * static_cast<uint32_t>(bn);
                for (int kb = 0; kb < P.kblocks; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1u;
                    if (!mbar_wait(&full[s], ph, abort_flag, p.status, tmo)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(stage_base + static_cast<size_t>(s) * stage_bytes);
                    const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t adesc = smem_desc_sw128(a_addr + kk * 2048, HALF_A, 1024);
                        const uint64_t bdesc = smem_desc_sw128(b_addr + kk * 32, 16, 1024);
                        tc_mma_bf16(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(&empty[s]);
                }
                if (!ok) break;
                tc_commit(&tfull[b]);
            }
            // drain: every MMA issued by this thread has completed before TMEM is freed
            tc_commit(drain);
            int dummy_abort = 0;
            mbar_wait(drain, 0, &dummy_abort, nullptr, 20000000ull);
        }
    } else {
        // ----------------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        uint32_t tc = 0, cc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const Tile T = decode(t);
            const ProbDev &P = p.prob[T.pi];
            const uint32_t b = tc & 1u, tph = (tc >> 1) & 1u;
            const bool ok = mbar_wait(&tfull[b], tph, abort_flag, p.status, tmo);
            if (!epi_all(ok)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * static_cast<uint32_t>(bn);
            const int nchunks = (T.nvalid + 15) / 16;
            if (MODE == MODE_UP) {
                const int i = T.mt * 64 + (q & 1) * 32 + lane;
                uint16_t *out = static_cast<uint16_t *>(P.out);
                for (int c = 0; c < nchunks; ++c, ++cc) {
                    float v[16];
                    __syncwarp();
                    tmem_ld16(tbase + 16 * c, v);
                    float *xb = xbuf + (cc & 1u) * (16 * 64);
                    if (q >= 2) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) xb[j * 64 + (q - 2) * 32 + lane] = v[j];
                    }
                    named_bar_sync(1, 128);
                    if (q < 2) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int n = 16 * c + j;
                            if (n < T.nvalid) {
                                const float u = xb[j * 64 + q * 32 + lane];
                                const float g = v[j];
                                const float h = g / (1.f + __expf(-g)) * u;
                                out[static_cast<size_t>(T.row0 + n) * P.out_ld + i] = f32_to_bf16_rn(h);
                            }
                        }
                    }
                }
            } else {
                const int col = T.mt * 128 + q * 32 + lane;
                const bool col_ok = col < P.out_cols;
                for (int c = 0; c < nchunks; ++c) {
                    float v[16];
                    __syncwarp();
                    tmem_ld16(tbase + 16 * c, v);
                    if (col_ok) {
                        if (P.out_fp32) {
                            float *out = static_cast<float *>(P.out);
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int n = 16 * c + j;
                                if (n < T.nvalid) out[static_cast<size_t>(T.row0 + n) * P.out_ld + col] = v[j];
                            }
                        } else {
                            uint16_t *out = static_cast<uint16_t *>(P.out);
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const int n = 16 * c + j;
                                if (n < T.nvalid)
                                    out[static_cast<size_t>(T.row0 + n) * P.out_ld + col] = f32_to_bf16_rn(v[j]);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[b]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
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
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 3-D bf16 weight tensor [n_groups][rows][cols] (cols contiguous), 64 x 64 boxes.
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
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 activation tensor [rows][cols], boxes of 64 columns x bn rows.
bool encode_act(CUtensorMap *m, const void *base, int rows, int cols, int bn)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(bn)};
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

size_t ffn_smem_bytes(int bn, int stages)
{
    return 1024 + static_cast<size_t>(stages) * (A_BYTES + bn * 128) + XCHG_FLOATS * 4 +
           (2 * stages + 5) * 8 + 16 + 4 * (MAX_GROUPS + 1) * 4;
}

int pick_stages(int bn)
{
    const size_t cap = 232448;   // max dynamic shared memory per block on sm_100/sm_103
    int s = 12;
    while (s > 2 && ffn_smem_bytes(bn, s) > cap) --s;
    return s;
}

}  // namespace

cudaError_t launch_ffn(const FfnProblem *probs, int n_probs, int H, const int *I_pp,
                       int token_hint, int *status, cudaStream_t s,
                       unsigned long long timeout_ns, int inject, cudaEvent_t mid_event)
{
    if (n_probs < 1 || n_probs > 2) return cudaErrorInvalidValue;
    const int bn = pick_bn(token_hint);
    const int stages = pick_stages(bn);
    const size_t smem = ffn_smem_bytes(bn, stages);
    int tcols = 32;
    while (tcols < 2 * bn) tcols <<= 1;

    FfnArgs up, dn;
    memset(&up, 0, sizeof up);
    memset(&dn, 0, sizeof dn);
    for (int pi = 0; pi < n_probs; ++pi) {
        const FfnProblem &P = probs[pi];
        const int I = I_pp[pi];
        if (!encode_weight(&up.mapA[pi], P.W1, P.n_groups, H, I) ||
            !encode_weight(&up.mapA3[pi], P.W3, P.n_groups, H, I) ||
            !encode_act(&up.mapB[pi], P.act, P.rows, H, bn) ||
            !encode_weight(&dn.mapA[pi], P.W2, P.n_groups, I, H) ||
            !encode_act(&dn.mapB[pi], P.h, P.rows, I, bn))
            return cudaErrorInvalidValue;
        dn.mapA3[pi] = dn.mapA[pi];
        ProbDev u{};
        u.offsets = P.offsets;
        u.n_groups = P.n_groups;
        u.dense_rows = P.dense_rows;
        u.n_mtiles = I / 64;
        u.kblocks = H / 64;
        u.out_ld = I;
        u.out_cols = I;
        u.out_fp32 = 0;
        u.out = P.h;
        up.prob[pi] = u;
        ProbDev d = u;
        d.n_mtiles = (H + 127) / 128;
        d.kblocks = I / 64;
        d.out_ld = H;
        d.out_cols = H;
        d.out_fp32 = P.out_fp32;
        d.out = P.out;
        dn.prob[pi] = d;
    }
    for (FfnArgs *a : {&up, &dn}) {
        a->n_probs = n_probs;
        a->bn = bn;
        a->stages = stages;
        a->tmem_cols = tcols;
        a->status = status;
        a->timeout_ns = timeout_ns;
        a->inject = inject;
    }
    cudaError_t err;
    err = ensure_smem(reinterpret_cast<const void *>(ffn_kernel<MODE_UP>), smem);
    if (err != cudaSuccess) return err;
    err = ensure_smem(reinterpret_cast<const void *>(ffn_kernel<MODE_DOWN>), smem);
    if (err != cudaSuccess) return err;
    const int grid = num_sms();
    ffn_kernel<MODE_UP><<<grid, NUM_THREADS, smem, s>>>(up);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    if (mid_event && (err = cudaEventRecord(mid_event, s)) != cudaSuccess) return err;
    ffn_kernel<MODE_DOWN><<<grid, NUM_THREADS, smem, s>>>(dn);
    return cudaGetLastError();
}

}  // namespace moe
