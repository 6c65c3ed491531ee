"""moe_router_topk_noalloc: the router for callers that cannot allocate device memory
(its scratch is a fixed array inside the library).  Checked through the C ABI against
moe_router_topk, which takes a caller-allocated workspace, and against the oracle, on
calls in a row on the router's different paths.

This file is collected last on purpose, so a run that stops at its first failure has
already run every other test; it sets up everything it needs itself and also passes
when run alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from expert_routed_ffn_router_gb300 import binding as B
from expert_routed_ffn_router_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
W_MAX_ABS = 1e-5          # routing-weight tolerance of the other parity tests


def _noalloc():
    lib = B.load()
    f = lib.moe_router_topk_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, I, I, I, I, P, P, P]
    f.restype = I
    return f


def _inputs(T, x_seed):
    w = synth.workload("decode", T=T, x_seed=x_seed)
    r = synth.routing_inputs(w)
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(DEV)
    return w, to(r["X"]), to(r["W_gate"]), torch.from_numpy(r["bias"]).to(DEV), r


def _with_workspace(w, X, Wg, bias):
    ws = torch.zeros(B.moe_workspace_bytes(w.T, w.H, w.E, w.K, w.I, w.Is), dtype=torch.uint8,
                     device=DEV)
    idx = torch.empty(w.T, w.K, dtype=torch.int32, device=DEV)
    wt = torch.empty(w.T, w.K, dtype=torch.float32, device=DEV)
    B.moe_router_topk(X, Wg, bias, w.K, idx, wt, ws)
    return idx, wt


def _without_workspace(f, w, X, Wg, bias):
    idx = torch.full((w.T, w.K), -7, dtype=torch.int32, device=DEV)
    wt = torch.full((w.T, w.K), -7.0, dtype=torch.float32, device=DEV)
    s = torch.cuda.current_stream()
    rc = f(ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(Wg.data_ptr()),
           ctypes.c_void_p(bias.data_ptr()), w.T, w.H, w.E, w.K,
           ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(wt.data_ptr()),
           ctypes.c_void_p(s.cuda_stream))
    assert rc == 0, B.moe_error_string(rc)
    return idx, wt


def test_noalloc_router_matches_workspace_router_twice():
    f = _noalloc()
    # calls in a row on different batches: a call must not see an earlier call's scratch.
    # 128, 77, 2048: the tile GEMM + one-warp-per-token finalise (2048 is the documented
    # upper end); 5 and 12, after those: the one-launch paths (one warp per expert up to 8
    # tokens, then the 16-token tile whose last CTA selects), which rely on the completion
    # counters being cleared in the shared array.
    for T, x_seed in ((128, 0), (77, 5), (2048, 9), (5, 11), (12, 13), (5, 17)):
        w, X, Wg, bias, r = _inputs(T, x_seed)
        ref_idx, ref_w = _with_workspace(w, X, Wg, bias)
        idx, wt = _without_workspace(f, w, X, Wg, bias)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx), T
        assert float((wt - ref_w).abs().max()) <= W_MAX_ABS, T
        # ... and against the oracle directly: bit-exact experts, weights within 1e-5
        idx_o, w_o = oracle.router(r["X"], r["W_gate"], r["bias"], w.K)
        assert np.array_equal(idx.cpu().numpy(), idx_o), T
        assert np.abs(wt.cpu().numpy().astype(np.float64) - w_o).max() <= W_MAX_ABS, T
    assert B.moe_router_topk_noalloc_status() == 0


def test_noalloc_router_rejects_shapes_beyond_its_scratch():
    f = _noalloc()
    w, X, Wg, bias, _ = _inputs(128, 0)
    # 65536 tokens need far more than the fixed 16 MiB of router scratch; rejected on the
    # host before anything is enqueued (the pointers are never dereferenced)
    rc = f(ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(Wg.data_ptr()),
           ctypes.c_void_p(bias.data_ptr()), 65536, w.H, w.E, w.K,
           ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(X.data_ptr()), None)
    assert rc == -2      # MOE_ERR_UNSUPPORTED_SHAPE
