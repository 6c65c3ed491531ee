// api.cu -- the C ABI of include/moe.h: argument validation, workspace layout and the
// kernel sequence of each entry point.  Everything is enqueued on the caller's stream;
// nothing here allocates, frees or synchronises (moe_read_status excepted).
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

namespace moe {

int num_sms()
{
    static std::atomic<int> cache[64];   // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

cudaError_t ensure_smem(const void *func, size_t bytes)
{
    // small table of (function, device) -> largest limit set so far; host threads making
    // their first calls at the same time share it, hence the lock
    struct Entry { const void *f; int dev; size_t bytes; };
    static Entry tab[64];
    static int n = 0;
    static std::mutex mu;
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (tab[i].f == func && tab[i].dev == dev && tab[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    for (int i = 0; i < n; ++i)
        if (tab[i].f == func && tab[i].dev == dev) { tab[i].bytes = bytes; return cudaSuccess; }
    if (n < 64) tab[n++] = Entry{func, dev, bytes};
    return cudaSuccess;
}

namespace {

constexpr size_t kHeader = 256;   // status word + reserved
unsigned long long g_wait_limit_ns = 1000000000ull;
int g_inject_stall = 0;
cudaEvent_t g_stage_events[6] = {};
bool g_stage_events_on = false;
int g_shared_side = -1;   // shared expert on the side stream: -1 by batch size, 0 never, 1 always
std::atomic<int> g_sync_status{0};   // debug mode: calls return their workspace's status word

// Up to this many tokens the router and the dispatch leave most of the GPU idle (their
// kernels wait on latency, not on SMs or HBM): the shared expert, which needs no routing,
// then runs beside them on a quarter of the SMs.  (The routed experts' launch takes the
// other SMs as soon as the dispatch is done; a quarter measured best of 1/8 .. 1: T=2
// 0.2458 ms with half of the SMs -> 0.2431 ms, T=64 1.618 -> 1.610, T=128 1.862 -> 1.855.)
constexpr int kSideMaxTokens = 128;
int side_ctas() { return num_sms() / 4 > 0 ? num_sms() / 4 : 1; }

// A stream of the library for the shared expert, forked from and joined back into the
// caller's stream with two events (capturable: the side stream joins a capture through the
// fork event).  One per host thread and device, created on first use and kept until the
// thread exits: calls from different threads (on different workspaces) never share the
// events, and the calls of one thread are sequential.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    bool tried = false;
};

// The side streams of one host thread; released when the thread exits (work still queued
// on a stream completes first: cudaStreamDestroy defers the release).  Errors are ignored:
// at process exit the runtime may already be gone.
struct SideStreams {
    SideStream tab[64];
    ~SideStreams()
    {
        for (SideStream &ss : tab) {
            if (ss.fork) cudaEventDestroy(ss.fork);
            if (ss.join) cudaEventDestroy(ss.join);
            if (ss.s) cudaStreamDestroy(ss.s);
        }
    }
};

SideStream *side_stream(cudaStream_t caller)
{
    thread_local SideStreams streams;
    SideStream *tab = streams.tab;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    SideStream &ss = tab[dev];
    if (!ss.tried) {
        // not created while the caller's stream is being captured (the call then keeps the
        // shared expert in the routed launch; a later call outside a capture creates it)
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(caller, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
            return nullptr;
        ss.tried = true;
        if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess)
            ss.s = nullptr;
    }
    return ss.s ? &ss : nullptr;
}

void record_stage(int i, cudaStream_t s)
{
    if (g_stage_events_on && g_stage_events[i]) cudaEventRecord(g_stage_events[i], s);
}

size_t al256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_common(int T, int H, int E, int K)
{
    if (T < 0 || H <= 0 || E <= 0 || K <= 0 || K > E) return MOE_ERR_INVALID_ARG;
    if (E > 1024 || K > 32 || H % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<long long>(T) * K >= (1ll << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

int check_ptrs(std::initializer_list<const void *> ps)
{
    for (const void *p : ps) {
        if (!p) return MOE_ERR_INVALID_ARG;
        if (!aligned(p, 16)) return MOE_ERR_MISALIGNED;
    }
    return MOE_OK;
}

int check_opt(const void *p) { return (p && !aligned(p, 16)) ? MOE_ERR_MISALIGNED : MOE_OK; }

int check_ws(const void *ws, size_t have, size_t need)
{
    if (!ws) return MOE_ERR_INVALID_ARG;
    if (!aligned(ws, 256)) return MOE_ERR_MISALIGNED;
    if (have < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return MOE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// moe_routing_t (NULL: defaults) -> validated options
int check_routing(const moe_routing_t *r, int E, int K, RoutingOpts &o)
{
    o = RoutingOpts{};
    if (!r) return MOE_OK;
    if (r->scoring != 0 && r->scoring != 1) return MOE_ERR_INVALID_ARG;
    if (r->renorm != 0 && r->renorm != 1) return MOE_ERR_INVALID_ARG;
    if (r->n_group < 1 || E % r->n_group != 0) return MOE_ERR_INVALID_ARG;
    const int G = E / r->n_group;
    if (r->topk_group < 1 || r->topk_group > r->n_group) return MOE_ERR_INVALID_ARG;
    if (r->group_top < 1 || r->group_top > G) return MOE_ERR_INVALID_ARG;
    if (static_cast<long long>(K) > static_cast<long long>(r->topk_group) * G) return MOE_ERR_INVALID_ARG;
    if (r->n_group > 32 || r->group_top > 2) return MOE_ERR_UNSUPPORTED_SHAPE;
    o.scoring = r->scoring;
    o.n_group = r->n_group;
    o.topk_group = r->n_group > 1 ? r->topk_group : 1;
    o.group_top = r->group_top;
    o.renorm = r->renorm;
    return MOE_OK;
}

struct RouterLayout {
    RouterPlan plan;
    RouterScratch scr;
    size_t bytes;
};
RouterLayout router_layout(int T, int H, int E, unsigned char *base)
{
    RouterLayout L{};
    L.plan = router_plan(T, H, E);
    size_t o = 0;
    L.scr.part = reinterpret_cast<float *>(base + o); o += L.plan.part_bytes;
    L.scr.xsq = reinterpret_cast<float *>(base + o); o += L.plan.xsq_bytes;
    L.scr.wsq = reinterpret_cast<float *>(base + o); o += L.plan.wsq_bytes;
    L.scr.cnt = reinterpret_cast<unsigned *>(base + o); o += L.plan.cnt_bytes;
    L.bytes = o;
    return L;
}

struct DispatchLayout {
    DispatchPlan plan;
    DispatchScratch scr;
    size_t bytes;
};
DispatchLayout dispatch_layout(int T, int E, unsigned char *base)
{
    DispatchLayout L{};
    L.plan = dispatch_plan(T, E);
    size_t o = 0;
    L.scr.smask = reinterpret_cast<uint32_t *>(base + o); o += L.plan.smask_bytes;
    L.scr.chunk_cnt = reinterpret_cast<int32_t *>(base + o); o += L.plan.ccnt_bytes;
    L.scr.chunk_base = reinterpret_cast<int32_t *>(base + o); o += L.plan.cbase_bytes;
    L.bytes = o;
    return L;
}

struct LayerLayout {
    RouterLayout r;
    DispatchLayout d;
    int32_t *offsets, *perm, *slot_pos;
    void *Xp, *h, *Yp, *hs;
    float *Ysh;
    // FP8 experts: E4M3 operands of the expert GEMMs and their block scales (fp32 2^k,
    // [blocks][fp8_scale_pitch(rows)]): permuted rows, token rows (shared expert), h, hs
    void *Xp8, *X8, *h8, *hs8;
    float *XpsT, *XsT, *hsT, *hssT;
    unsigned *ready, *ready_sh;   // readiness counters: the FFN launch, the side launch
    moe_workspace_layout_t at;    // byte offsets of the intermediates inside the workspace
    size_t bytes;
};
LayerLayout layer_layout(const moe_shape_t &s, unsigned char *ws)
{
    LayerLayout L{};
    const size_t TK = static_cast<size_t>(s.T) * s.K;
    size_t o = kHeader;
    L.r = router_layout(s.T, s.H, s.E, ws ? ws + o : nullptr); o += L.r.bytes;
    L.d = dispatch_layout(s.T, s.E, ws ? ws + o : nullptr); o += L.d.bytes;
    size_t at = 0;
    auto take = [&](size_t b) {
        unsigned char *p = ws ? ws + o : nullptr;
        at = o;
        o += al256(b);
        return p;
    };
    L.offsets = reinterpret_cast<int32_t *>(take((s.E + 1) * sizeof(int32_t)));
    L.at.offsets = at;
    L.perm = reinterpret_cast<int32_t *>(take(TK * sizeof(int32_t)));
    L.at.perm = at;
    L.slot_pos = reinterpret_cast<int32_t *>(take(TK * sizeof(int32_t)));
    L.at.slot_pos = at;
    L.Xp = take(TK * s.H * 2);
    L.at.Xp = at;
    L.h = take(TK * s.I * 2);
    L.at.h = at;
    L.Yp = take(TK * s.H * 2);
    L.at.Yp = at;
    L.hs = take(static_cast<size_t>(s.T) * s.I_shared * 2);
    L.Ysh = reinterpret_cast<float *>(take(s.I_shared > 0 ? static_cast<size_t>(s.T) * s.H * 4 : 0));
    L.at.Ysh = at;
    {
        const size_t pT = static_cast<size_t>(fp8_scale_pitch(s.T));
        const size_t pTK = static_cast<size_t>(fp8_scale_pitch(static_cast<long long>(TK)));
        const size_t bH = (s.H + 127) / 128, bI = (s.I + 127) / 128, bIs = (s.I_shared + 127) / 128;
        L.Xp8 = take(TK * s.H);
        L.XpsT = reinterpret_cast<float *>(take(bH * pTK * 4));
        L.X8 = take(static_cast<size_t>(s.T) * s.H);
        L.XsT = reinterpret_cast<float *>(take(bH * pT * 4));
        L.h8 = take(TK * s.I);
        L.hsT = reinterpret_cast<float *>(take(bI * pTK * 4));
        L.hs8 = take(static_cast<size_t>(s.T) * s.I_shared);
        L.hssT = reinterpret_cast<float *>(take(bIs * pT * 4));
    }
    
    L.ready = reinterpret_cast<unsigned *>(
        take(ffn_ready_slots(static_cast<long long>(TK) + s.T, s.E + 1) * sizeof(unsigned)));
    L.ready_sh = reinterpret_cast<unsigned *>(
        take(s.I_shared > 0 ? ffn_ready_slots(s.T, 1) * sizeof(unsigned) : 0));
    L.bytes = o;
    L.at.bytes = o;
    return L;
}

int check_shape(const moe_shape_t *s)
{
    if (!s) return MOE_ERR_INVALID_ARG;
    int rc = check_common(s->T, s->H, s->E, s->K);
    if (rc) return rc;
    if (s->I <= 0 || s->I_shared < 0) return MOE_ERR_INVALID_ARG;
    if (s->I % 64 != 0 || s->I_shared % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

// The layer on bf16 expert weights (wt) or FP8 ones (w8: E4M3 with 128 x 128 power-of-two
// block scales; the token rows and h are then quantised on the fly in vectors of 128).
int layer_forward(const moe_shape_t *shape, const moe_weights_t *wt, const moe_weights_fp8_t *w8,
                  const moe_routing_t *routing, const void *X, float *Y, int32_t *topk_idx,
                  float *topk_w, int32_t *counts, int32_t *affinity, void *ws, size_t ws_bytes,
                  void *stream)
{
    int rc = check_shape(shape);
    if (rc) return rc;
    const moe_shape_t s = *shape;
    RoutingOpts ro;
    if ((rc = check_routing(routing, s.E, s.K, ro))) return rc;
    const bool fp8 = w8 != nullptr;
    const void *W_gate = fp8 ? w8->W_gate : wt->W_gate;
    const float *bias = fp8 ? w8->bias : static_cast<const float *>(wt->bias);
    const void *W1 = fp8 ? w8->W1 : wt->W1, *W3 = fp8 ? w8->W3 : wt->W3, *W2 = fp8 ? w8->W2 : wt->W2;
    const void *W1s = fp8 ? w8->W1s : wt->W1s, *W3s = fp8 ? w8->W3s : wt->W3s,
               *W2s = fp8 ? w8->W2s : wt->W2s;
    if ((rc = check_ptrs({X, Y, topk_idx, topk_w, counts, W_gate, bias, W1, W3, W2}))) return rc;
    if (s.I_shared > 0 && (rc = check_ptrs({W1s, W3s, W2s}))) return rc;
    if (fp8) {
        if (s.H % 128 || s.I % 128 || s.I_shared % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
        if (s.H > 16384 || s.I > 16384 || s.I_shared > 16384) return MOE_ERR_UNSUPPORTED_SHAPE;
        if (!w8->S1 || !w8->S3 || !w8->S2) return MOE_ERR_INVALID_ARG;
        if (s.I_shared > 0 && (!w8->S1s || !w8->S3s || !w8->S2s)) return MOE_ERR_INVALID_ARG;
    }
    if ((rc = check_opt(affinity))) return rc;
    unsigned char *w = static_cast<unsigned char *>(ws);
    const LayerLayout L = layer_layout(s, w);
    if ((rc = check_ws(ws, ws_bytes, L.bytes))) return rc;
    if (s.T == 0) return MOE_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int *status = static_cast<int *>(ws);

    FfnProblem P[2]{};
    int Ipp[2] = {s.I, s.I_shared};
    P[0].offsets = L.offsets;
    P[0].n_groups = s.E;
    P[0].rows = s.T * s.K;
    P[0].W1 = W1; P[0].W3 = W3; P[0].W2 = W2;
    P[0].h = L.h;
    P[0].out = L.Yp;
    P[0].out_fp32 = 0;
    if (fp8) {
        P[0].fp8 = 1;
        P[0].S1 = w8->S1; P[0].S3 = w8->S3; P[0].S2 = w8->S2;
        P[0].act_s = L.XpsT;
        P[0].h8 = L.h8;
        P[0].h_s = L.hsT;
    }
    int n_probs = 1;
    if (s.I_shared > 0) {
        P[1].offsets = nullptr;
        P[1].n_groups = 1;
        P[1].rows = s.T;
        P[1].dense_rows = s.T;
        P[1].W1 = W1s; P[1].W3 = W3s; P[1].W2 = W2s;
        P[1].h = L.hs;
        P[1].out = L.Ysh;
        P[1].out_fp32 = 1;
        if (fp8) {
            P[1].fp8 = 1;
            P[1].S1 = w8->S1s; P[1].S3 = w8->S3s; P[1].S2 = w8->S2s;
            P[1].act_s = L.XsT;
            P[1].h8 = L.hs8;
            P[1].h_s = L.hssT;
        }
        n_probs = 2;
    }

    // shared expert beside the router and the dispatch (bf16 weights, small batches)
    SideStream *side = nullptr;
    if (!fp8 && s.I_shared > 0 && (g_shared_side == 1 || (g_shared_side < 0 && s.T <= kSideMaxTokens)))
        side = side_stream(st);
    if (side) {
        P[1].act = X;
        if (cudaEventRecord(side->fork, st) != cudaSuccess ||
            cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (launch_ffn(&P[1], 1, s.H, &Ipp[1], s.T, L.ready_sh, false, status, side->s,
                       g_wait_limit_ns, g_inject_stall, nullptr, -1, side_ctas()) != cudaSuccess ||
            cudaEventRecord(side->join, side->s) != cudaSuccess)
            return MOE_ERR_CUDA;
        n_probs = 1;
    }

    record_stage(0, st);
    cudaError_t e = launch_router(X, W_gate, bias, s.T, s.H, s.E, s.K, topk_idx, topk_w,
                                  L.r.plan, L.r.scr, status, st, &ro);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    record_stage(1, st);
    // the dispatch tail also zeroes the FFN's readiness counters
    const size_t n_ready = ffn_ready_slots(static_cast<long long>(s.T) * s.K + s.T, s.E + 1);
    e = launch_dispatch(X, topk_idx, s.T, s.H, s.E, s.K, counts, L.offsets, L.perm, L.slot_pos,
                        L.Xp, affinity, L.d.plan, L.d.scr, L.ready, n_ready, status, st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    const long long TK = static_cast<long long>(s.T) * s.K;
    if (fp8) {
        // the expert GEMMs' inputs as E4M3 rows with a scale per 128 along H: the permuted
        // rows and (shared expert) the token rows
        e = launch_quant_rows_e4m3(L.Xp, TK, s.H, L.Xp8, L.XpsT, fp8_scale_pitch(TK), st);
        if (e == cudaSuccess && s.I_shared > 0)
            e = launch_quant_rows_e4m3(X, s.T, s.H, L.X8, L.XsT, fp8_scale_pitch(s.T), st);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    record_stage(2, st);

    P[0].act = fp8 ? L.Xp8 : L.Xp;
    if (s.I_shared > 0 && !side) P[1].act = fp8 ? L.X8 : X;
    long long hint = static_cast<long long>(s.T) * s.K / s.E;
    if (hint < 1) hint = 1;
    if (!fp8) {
        e = launch_ffn(P, n_probs, s.H, Ipp, static_cast<int>(hint), L.ready, true, status, st,
                       g_wait_limit_ns, g_inject_stall, g_stage_events_on ? g_stage_events[3] : nullptr);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    } else {
        // up projections, h (bf16) quantised to E4M3 in vectors of 128 along I, then the down
        // projections
        e = launch_ffn(P, n_probs, s.H, Ipp, static_cast<int>(hint), L.ready, true, status, st,
                       g_wait_limit_ns, g_inject_stall, nullptr, 0);
        if (e == cudaSuccess) e = launch_quant_rows_e4m3(L.h, TK, s.I, L.h8, L.hsT, fp8_scale_pitch(TK), st);
        if (e == cudaSuccess && s.I_shared > 0)
            e = launch_quant_rows_e4m3(L.hs, s.T, s.I_shared, L.hs8, L.hssT, fp8_scale_pitch(s.T), st);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        record_stage(3, st);
        e = launch_ffn(P, n_probs, s.H, Ipp, static_cast<int>(hint), L.ready, true, status, st,
                       g_wait_limit_ns, g_inject_stall, nullptr, 1);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    record_stage(4, st);
    if (side && cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess) return MOE_ERR_CUDA;
    e = launch_combine(L.Yp, L.slot_pos, topk_w, s.I_shared > 0 ? L.Ysh : nullptr, s.T, s.H,
                       s.K, Y, st);
    record_stage(5, st);
    return cuda_status(e);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(const moe_shape_t *shape)
{
    if (check_shape(shape) != MOE_OK) return 0;
    return layer_layout(*shape, nullptr).bytes;
}

int moe_workspace_layout(const moe_shape_t *shape, moe_workspace_layout_t *out)
{
    if (!out) return MOE_ERR_INVALID_ARG;
    const int rc = check_shape(shape);
    if (rc) return rc;
    *out = layer_layout(*shape, nullptr).at;
    return MOE_OK;
}

const char *moe_error_string(int status)
{
    switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_MISALIGNED: return "misaligned pointer";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "bounded device-side wait ran out";
    case MOE_ERR_NOT_IMPLEMENTED: return "not implemented";
    default: return "unknown status";
    }
}

int moe_read_status(void *ws, void *stream)
{
    if (!ws) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, sizeof v, s) != cudaSuccess) return MOE_ERR_CUDA;
    return v;
}

void moe_debug_set_sync_status(int on)
{
    g_sync_status.store(on ? 1 : 0, std::memory_order_relaxed);
}

// Debug mode: after a call enqueued work without error, synchronise its stream and return
// the workspace's status word (read and reset as by moe_read_status) -- unless nothing was
// enqueued (an empty batch) or the stream is being captured into a graph, which cannot be
// synchronised.
static int debug_status(int rc, void *ws, void *stream, bool enqueued = true)
{
    if (rc != MOE_OK || !enqueued || g_sync_status.load(std::memory_order_relaxed) == 0)
        return rc;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return rc;
    return moe_read_status(ws, stream);
}

void moe_debug_set_wait_limit(unsigned long long limit_ns, int inject_stall)
{
    g_wait_limit_ns = limit_ns ? limit_ns : 1000000000ull;
    g_inject_stall = inject_stall;
}

void moe_debug_set_shared_side(int mode)
{
    g_shared_side = mode == 0 || mode == 1 ? mode : -1;
}

void moe_debug_set_ffn_variant(int variant)
{
    moe::set_ffn_variant(variant == 1 || variant == 2 ? variant : 0);
}

void moe_debug_set_stage_events(void *const *events, int n)
{
    g_stage_events_on = events != nullptr && n >= 6;
    for (int i = 0; i < 6; ++i)
        g_stage_events[i] = g_stage_events_on ? static_cast<cudaEvent_t>(events[i]) : nullptr;
}

int moe_router_topk(const void *X, const void *W_gate, const float *bias, int T, int H, int E,
                    int K, int32_t *topk_idx, float *topk_w, void *ws, size_t ws_bytes,
                    void *stream)
{
    return moe_router_topk_ex(X, W_gate, bias, T, H, E, K, nullptr, topk_idx, topk_w, ws,
                              ws_bytes, stream);
}

int moe_router_topk_ex(const void *X, const void *W_gate, const float *bias, int T, int H,
                       int E, int K, const moe_routing_t *routing, int32_t *topk_idx,
                       float *topk_w, void *ws, size_t ws_bytes, void *stream)
{
    int rc = check_common(T, H, E, K);
    if (rc) return rc;
    RoutingOpts ro;
    if ((rc = check_routing(routing, E, K, ro))) return rc;
    if ((rc = check_ptrs({X, W_gate, bias, topk_idx, topk_w}))) return rc;
    unsigned char *w = static_cast<unsigned char *>(ws);
    const RouterLayout L = router_layout(T, H, E, w ? w + kHeader : nullptr);
    if ((rc = check_ws(ws, ws_bytes, kHeader + L.bytes))) return rc;
    if (T == 0) return MOE_OK;
    return debug_status(cuda_status(launch_router(X, W_gate, bias, T, H, E, K, topk_idx, topk_w,
                                                  L.plan, L.scr, static_cast<int *>(ws),
                                                  static_cast<cudaStream_t>(stream), &ro)),
                        ws, stream);
}

int moe_dispatch(const void *X, const int32_t *topk_idx, int T, int H, int E, int K,
                 int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *slot_pos, void *Xp,
                 int32_t *affinity, void *ws, size_t ws_bytes, void *stream)
{
    int rc = check_common(T, H, E, K);
    if (rc) return rc;
    if ((rc = check_ptrs({X, topk_idx, counts, offsets, perm, slot_pos, Xp}))) return rc;
    if ((rc = check_opt(affinity))) return rc;
    unsigned char *w = static_cast<unsigned char *>(ws);
    const DispatchLayout L = dispatch_layout(T, E, w ? w + kHeader : nullptr);
    if ((rc = check_ws(ws, ws_bytes, kHeader + L.bytes))) return rc;
    if (T == 0) return MOE_OK;
    return debug_status(cuda_status(launch_dispatch(X, topk_idx, T, H, E, K, counts, offsets,
                                                    perm, slot_pos, Xp, affinity, L.plan, L.scr,
                                                    nullptr, 0, static_cast<int *>(ws),
                                                    static_cast<cudaStream_t>(stream))),
                        ws, stream);
}

size_t moe_expert_ffn_workspace_bytes(int rows, int n_groups, int I)
{
    if (rows < 0 || n_groups <= 0 || n_groups > 1024 || I <= 0) return 0;
    return kHeader + al256(static_cast<size_t>(rows) * I * 2) +
           al256(ffn_ready_slots(rows, n_groups) * sizeof(unsigned));
}

int moe_expert_ffn(const void *Xp, const int32_t *offsets, int n_groups, int rows, int H, int I,
                   const void *W1, const void *W3, const void *W2, void *Yp, int out_fp32,
                   void *ws, size_t ws_bytes, void *stream)
{
    if (n_groups <= 0 || rows < 0 || H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
    if (n_groups > 1024 || H % 64 != 0 || I % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (out_fp32 != 0 && out_fp32 != 1) return MOE_ERR_INVALID_ARG;
    int rc = check_ptrs({Xp, offsets, W1, W3, W2, Yp});
    if (rc) return rc;
    const size_t hbytes = al256(static_cast<size_t>(rows) * I * 2);
    const size_t rbytes = al256(ffn_ready_slots(rows, n_groups) * sizeof(unsigned));
    if ((rc = check_ws(ws, ws_bytes, kHeader + hbytes + rbytes))) return rc;
    if (rows == 0) return MOE_OK;
    FfnProblem P{};
    P.act = Xp;
    P.offsets = offsets;
    P.n_groups = n_groups;
    P.rows = rows;
    P.W1 = W1; P.W3 = W3; P.W2 = W2;
    P.h = static_cast<unsigned char *>(ws) + kHeader;
    P.out = Yp;
    P.out_fp32 = out_fp32;
    const int hint = rows / n_groups > 0 ? rows / n_groups : 1;
    unsigned *ready = reinterpret_cast<unsigned *>(static_cast<unsigned char *>(ws) + kHeader + hbytes);
    return debug_status(cuda_status(launch_ffn(&P, 1, H, &I, hint, ready, false,
                                               static_cast<int *>(ws),
                                               static_cast<cudaStream_t>(stream), g_wait_limit_ns,
                                               g_inject_stall, nullptr)),
                        ws, stream);
}

int moe_combine(const void *Yp, const int32_t *slot_pos, const float *topk_w, const float *Ysh,
                int T, int H, int K, float *Y, void *stream)
{
    if (T < 0 || H <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
    if (H % 64 != 0 || K > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
    int rc = check_ptrs({Yp, slot_pos, topk_w, Y});
    if (rc) return rc;
    if ((rc = check_opt(Ysh))) return rc;
    if (T == 0) return MOE_OK;
    return cuda_status(launch_combine(Yp, slot_pos, topk_w, Ysh, T, H, K, Y,
                                      static_cast<cudaStream_t>(stream)));
}

int moe_layer_forward(const moe_shape_t *shape, const moe_weights_t *wt, const void *X, float *Y,
                      int32_t *topk_idx, float *topk_w, int32_t *counts, int32_t *affinity,
                      void *ws, size_t ws_bytes, void *stream)
{
    return moe_layer_forward_ex(shape, wt, nullptr, X, Y, topk_idx, topk_w, counts, affinity,
                                ws, ws_bytes, stream);
}

int moe_layer_forward_ex(const moe_shape_t *shape, const moe_weights_t *wt,
                         const moe_routing_t *routing, const void *X, float *Y,
                         int32_t *topk_idx, float *topk_w, int32_t *counts, int32_t *affinity,
                         void *ws, size_t ws_bytes, void *stream)
{
    if (!wt) return MOE_ERR_INVALID_ARG;
    return debug_status(layer_forward(shape, wt, nullptr, routing, X, Y, topk_idx, topk_w, counts,
                                      affinity, ws, ws_bytes, stream),
                        ws, stream, shape && shape->T > 0);
}

int moe_layer_forward_fp8(const moe_shape_t *shape, const moe_weights_fp8_t *w8,
                          const moe_routing_t *routing, const void *X, float *Y,
                          int32_t *topk_idx, float *topk_w, int32_t *counts, int32_t *affinity,
                          void *ws, size_t ws_bytes, void *stream)
{
    if (!w8) return MOE_ERR_INVALID_ARG;
    return debug_status(layer_forward(shape, nullptr, w8, routing, X, Y, topk_idx, topk_w, counts,
                                      affinity, ws, ws_bytes, stream),
                        ws, stream, shape && shape->T > 0);
}

int moe_quantize_weight_fp8(const void *W, int G, int R, int C, void *Wq, int32_t *S,
                            void *stream)
{
    if (G < 0 || R <= 0 || C <= 0) return MOE_ERR_INVALID_ARG;
    if (R % 128 || C % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    int rc = check_ptrs({W, Wq});
    if (rc) return rc;
    if (!S) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(S) % 4) return MOE_ERR_MISALIGNED;
    if (G == 0) return MOE_OK;
    return cuda_status(launch_quant_weight(W, G, R, C, Wq, S, static_cast<cudaStream_t>(stream)));
}

int moe_quantize_rows_fp8(const void *in, long long rows, int n, void *out, void *stream)
{
    if (rows < 0 || n <= 0) return MOE_ERR_INVALID_ARG;
    if (n % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    int rc = check_ptrs({in, out});
    if (rc) return rc;
    if (rows == 0) return MOE_OK;
    return cuda_status(launch_quant_rows(in, rows, n, out, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
