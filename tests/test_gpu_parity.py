"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded
inputs.  Integer outputs (top-k indices, counts, offsets, permutation, slot positions,
affinity) must be bit-exact; routing weights within 1e-5; Y within relative Frobenius
5e-3 and max-abs 3e-2."""
import numpy as np
import pytest
import torch

import oracle
from expert_routed_ffn_router_gb300 import binding as B
from expert_routed_ffn_router_gb300 import synth

from gpu_common import (DEV, W_MAX_ABS, Y_MAX_ABS, Y_REL_FROB, Problem, bits, check_layer,
                        host_to_device_bf16, rel_frob)

pytestmark = pytest.mark.gpu


def _ws(nbytes):
    return torch.zeros(nbytes, dtype=torch.uint8, device=DEV)


# --------------------------------------------------------------------------- whole layer
def test_tiny_layer():
    r = check_layer(Problem(synth.workload("tiny")))
    assert r["rel_frob"] < 2e-3


@pytest.mark.parametrize("T,H,E,K,I,Is", [
    (1, 256, 16, 2, 128, 128),      # a single token: 14 experts receive nothing
    (3, 256, 16, 2, 128, 128),      # tiny batch: 3 of a 4-token router batch
    (6, 256, 16, 2, 128, 128),      # 6 of an 8-token router batch
    (37, 256, 16, 2, 128, 128),     # ragged token tail
    (300, 192, 40, 5, 192, 64),     # H % 128 == 64, E not a multiple of 32, K = 5
    (130, 128, 8, 8, 64, 0),        # K == E (every expert, order only), no shared expert
    (513, 256, 64, 6, 256, 128),    # several dispatch chunks
    (513, 256, 8, 6, 128, 128),     # 385 rows per expert: 256-row token tiles
    (700, 192, 16, 4, 192, 64),     # 256-row tiles, odd weight-tile counts (3 up, 2 down)
    (128, 128, 16, 2, 128, 0),      # 16 rows per expert: 128-row token tiles
    (50, 128, 8, 1, 64, 64),        # top-1 routing
    (20, 64, 1, 1, 64, 0),          # a single expert (E = K = 1), H = I = 64
    (5, 128, 1024, 8, 64, 0),       # the largest E: a batch the one-launch router would
                                    # take, whose finalising CTA cannot hold 1024 experts
    (40, 128, 1024, 4, 64, 64),     # the largest E on the tile + finalise path
    (2100, 64, 1024, 2, 64, 0),     # the largest E at a size of the one-launch 16-token tile
    (100, 128, 64, 32, 64, 0),      # the largest K
    (30, 128, 48, 32, 64, 64),      # the largest K, E not a multiple of 32
])
def test_ragged_shapes(T, H, E, K, I, Is):
    w = synth.Workload("rag", T=T, H=H, E=E, K=K, I=I, Is=Is, seed=T, x_seed=T + 1)
    check_layer(Problem(w))


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("T,H,E,K,I,Is", [
    (37, 256, 16, 2, 128, 128),     # 32-row tiles (a pair splits them 16 + 16)
    (300, 192, 40, 5, 192, 64),     # pair tiles past the last weight column (I, H % 256)
    (130, 128, 8, 8, 64, 0),        # I = 64: the odd CTA of every up tile is all padding
    (513, 256, 8, 6, 128, 128),     # 256-row token tiles, ragged last tile per expert
    (700, 192, 16, 4, 192, 64),
])
def test_ffn_variants_single_cta_and_cta_pair(T, H, E, K, I, Is, variant):
    w = synth.Workload("var", T=T, H=H, E=E, K=K, I=I, Is=Is, seed=T + 5, x_seed=T + 6)
    B.moe_debug_set_ffn_variant(variant)
    try:
        check_layer(Problem(w))
    finally:
        B.moe_debug_set_ffn_variant(0)


def test_exact_ties_duplicate_gate_rows():
    w = synth.workload("tiny", T=64)
    r = synth.routing_inputs(w)
    for a, b in ((1, 9), (4, 5), (0, 15)):
        r["W_gate"][b] = r["W_gate"][a]
        r["bias"][b] = r["bias"][a]
    r["bias"][4] = r["bias"][5] = 2.0     # the tied pair is the top-2 of every token
    res = check_layer(Problem(w, routing=r))
    both = [row for row in res["idx"].tolist() if 4 in row and 5 in row]
    assert both and all(row.index(4) < row.index(5) for row in both)


def test_near_ties_take_the_refine_path():
    # gate rows that differ in one bf16 ulp of one element: selection scores a few 1e-6
    # apart, far inside the fp32 error bound, so the exact order must come from the refine
    w = synth.workload("tiny", T=96)
    r = synth.routing_inputs(w)
    for a, b in ((2, 3), (7, 11), (12, 13)):
        r["W_gate"][b] = r["W_gate"][a]
        r["W_gate"][b, 17] = r["W_gate"][a, 17] + 1
        r["bias"][b] = r["bias"][a]
    check_layer(Problem(w, routing=r))


def test_one_expert_takes_every_token():
    w = synth.workload("tiny", T=200)
    r = synth.routing_inputs(w)
    r["bias"][3] = 10.0
    res = check_layer(Problem(w, routing=r))
    assert res["disp"]["counts"][3] == w.T


@pytest.mark.parametrize("side", [0, 1])
def test_deterministic_and_graph_capture(side):
    # side = 1: the shared expert on the library's side stream, which joins the capture
    B.moe_debug_set_shared_side(side)
    try:
        _deterministic_and_graph_capture()
    finally:
        B.moe_debug_set_shared_side(-1)


@pytest.mark.parametrize("side", [0, 1])
@pytest.mark.parametrize("T", [3, 40, 300])
def test_shared_expert_in_the_routed_launch_or_beside_the_router(side, T):
    w = synth.Workload("side", T=T, H=256, E=16, K=4, I=128, Is=192, seed=T + 51, x_seed=T + 52)
    B.moe_debug_set_shared_side(side)
    try:
        check_layer(Problem(w))
    finally:
        B.moe_debug_set_shared_side(-1)


def test_concurrent_calls_from_two_host_threads():
    # two host threads, each with its own layer (workspace) and stream, run the layer at the
    # same time; each thread's shared expert takes its own side stream, so the results are
    # those of the calls run one after the other
    import threading
    p = Problem(synth.workload("tiny", T=40))
    layers = [B.MoELayer(p.dev, p.w.T, p.w.K) for _ in range(2)]
    Xs = [p.X, p.X.flip(0).contiguous()]
    ref = []
    for layer, X in zip(layers, Xs):
        layer.forward(X)
        torch.cuda.synchronize()
        ref.append(layer.Y.clone())
    streams = [torch.cuda.Stream() for _ in range(2)]
    errors = []

    def run(i):
        try:
            torch.cuda.set_device(0)
            for _ in range(50):
                layers[i].forward(Xs[i], stream=streams[i])
        except Exception as exc:          # reported below, on the main thread
            errors.append(exc)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for layer, r in zip(layers, ref):
        assert torch.equal(layer.Y, r)
        assert layer.status() == 0


def test_first_call_of_a_host_thread_inside_a_graph_capture():
    # a host thread whose first layer call is captured: its side stream is not created
    # during the capture (that call keeps the shared expert in the routed launch), and the
    # replay gives what an ordinary call gives
    import threading
    p = Problem(synth.workload("tiny", T=24))
    layer = B.MoELayer(p.dev, p.w.T, p.w.K)
    layer.forward(p.X)                      # shared-memory limits raised outside the capture
    B.moe_debug_set_shared_side(0)          # the reference in the placement the capture takes
    try:
        layer.forward(p.X)
        torch.cuda.synchronize()
    finally:
        B.moe_debug_set_shared_side(-1)
    ref = layer.Y.clone()
    out = {}

    def run():
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            X2 = p.X.clone()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    layer.forward(X2, stream=s)
                layer.Y.zero_()
                g.replay()
            torch.cuda.synchronize()
            out["y"] = layer.Y.clone()
        except Exception as exc:          # reported below, on the main thread
            out["err"] = exc

    th = threading.Thread(target=run)
    th.start()
    th.join()
    assert "err" not in out, out.get("err")
    assert torch.equal(out["y"], ref)
    assert layer.status() == 0


def _deterministic_and_graph_capture():
    p = Problem(synth.workload("tiny", T=77))
    layer = B.MoELayer(p.dev, p.w.T, p.w.K)
    layer.forward(p.X)
    torch.cuda.synchronize()
    y1 = layer.Y.clone()
    layer.forward(p.X)
    torch.cuda.synchronize()
    assert torch.equal(y1, layer.Y)
    # capture the whole layer in a CUDA graph and replay it on new activations
    s = torch.cuda.Stream()
    X2 = p.X.clone()
    with torch.cuda.stream(s):
        layer.forward(X2, stream=s)            # warm-up on the capture stream
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            layer.forward(X2, stream=s)
    torch.cuda.synchronize()
    Xn = host_to_device_bf16(synth.f32_to_bf16_bits(
        np.random.default_rng(5).standard_normal((p.w.T, p.w.H)).astype(np.float32)))
    X2.copy_(Xn)
    g.replay()
    torch.cuda.synchronize()
    y_graph = layer.Y.clone()
    layer.forward(Xn)
    torch.cuda.synchronize()
    assert torch.equal(y_graph, layer.Y)
    assert layer.status() == 0


# --------------------------------------------------------------------- separate stages
def test_stages_separately_tiny():
    w = synth.workload("tiny", T=45)
    p = Problem(w)
    T, H, E, K, I = w.T, w.H, w.E, w.K, w.I
    ws = _ws(B.moe_workspace_bytes(T, H, E, K, I, w.Is))
    idx = torch.empty(T, K, dtype=torch.int32, device=DEV)
    wt = torch.empty(T, K, dtype=torch.float32, device=DEV)
    B.moe_router_topk(p.X, p.dev["W_gate"], p.dev["bias"], K, idx, wt, ws)
    idx_o, w_o = p.oracle_routing()
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    assert np.abs(wt.cpu().numpy() - w_o).max() <= W_MAX_ABS

    # dispatch fed the oracle's routing (no GPU-made input reaches the oracle)
    idx_in = torch.from_numpy(idx_o).to(DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * K, dtype=torch.int32, device=DEV)
    slot = torch.empty(T, K, dtype=torch.int32, device=DEV)
    Xp = torch.empty(T * K, H, dtype=torch.bfloat16, device=DEV)
    aff = torch.empty(E, E, dtype=torch.int32, device=DEV)
    B.moe_dispatch(p.X, idx_in, E, counts, offsets, perm, slot, Xp, aff, ws)
    d = oracle.dispatch(idx_o, E)
    for name, t in (("counts", counts), ("offsets", offsets), ("perm", perm),
                    ("slot_pos", slot), ("affinity", aff)):
        assert np.array_equal(t.cpu().numpy().reshape(d[name].shape), d[name]), name
    assert np.array_equal(bits(Xp), p.routing["X"][d["perm"]])

    # expert FFN on the oracle's permutation of X
    Xp_h = p.routing["X"][d["perm"]]
    Xp_in = host_to_device_bf16(Xp_h)
    off_in = torch.from_numpy(d["offsets"]).to(DEV)
    Yp = torch.empty(T * K, H, dtype=torch.float32, device=DEV)
    B.moe_expert_ffn(Xp_in, off_in, E, p.dev["W1"], p.dev["W3"], p.dev["W2"], Yp, ws)
    torch.cuda.synchronize()
    rows_e = np.searchsorted(d["offsets"], np.arange(T * K), side="right") - 1
    y_o = oracle.expert_rows(list(Xp_h), [p.host_w["W1"][e] for e in rows_e],
                             [p.host_w["W3"][e] for e in rows_e],
                             [p.host_w["W2"][e] for e in rows_e], H, I)
    y_g = Yp.cpu().numpy().astype(np.float64)
    assert rel_frob(y_g, y_o) <= Y_REL_FROB and np.abs(y_g - y_o).max() <= Y_MAX_ABS

    # combine on a synthetic Yp and the oracle's slots, weights rounded to fp32 on both sides
    rng = np.random.default_rng(3)
    Yp_h = synth.f32_to_bf16_bits(rng.standard_normal((T * K, H)).astype(np.float32))
    Ysh_h = rng.standard_normal((T, H)).astype(np.float32)
    w32 = w_o.astype(np.float32)
    Y = torch.empty(T, H, dtype=torch.float32, device=DEV)
    B.moe_combine(host_to_device_bf16(Yp_h), torch.from_numpy(d["slot_pos"]).to(DEV),
                  torch.from_numpy(w32).to(DEV), torch.from_numpy(Ysh_h).to(DEV), Y)
    Y_o = oracle.combine(Yp_h, d["slot_pos"], w32.astype(np.float64), Ysh_h.astype(np.float64))
    assert np.abs(Y.cpu().numpy() - Y_o).max() <= 1e-5
    assert B.moe_read_status(ws) == 0


def test_shared_expert_alone_is_a_dense_group():
    w = synth.workload("tiny", T=70)
    p = Problem(w)
    T, H, Is = w.T, w.H, w.Is
    ws = _ws(B.moe_workspace_bytes(T, H, 1, 1, Is, 0))
    off = torch.tensor([0, T], dtype=torch.int32, device=DEV)
    Y = torch.empty(T, H, dtype=torch.float32, device=DEV)
    B.moe_expert_ffn(p.X, off, 1, p.dev["W1s"].unsqueeze(0).contiguous(),
                     p.dev["W3s"].unsqueeze(0).contiguous(),
                     p.dev["W2s"].unsqueeze(0).contiguous(), Y, ws)
    torch.cuda.synchronize()
    X = p.routing["X"]
    y_o = oracle.expert_rows(list(X), [p.host_w["W1s"]] * T, [p.host_w["W3s"]] * T,
                             [p.host_w["W2s"]] * T, H, Is)
    assert rel_frob(Y.cpu().numpy().astype(np.float64), y_o) <= Y_REL_FROB


# ------------------------------------------------------------------ bounded waits
def test_bounded_wait_reports_timeout_and_context_survives():
    w = synth.workload("tiny", T=40)
    p = Problem(w)
    layer = B.MoELayer(p.dev, w.T, w.K)
    try:
        B.moe_debug_set_wait_limit(50_000_000, inject_stall=1)    # 50 ms
        layer.forward(p.X)
        torch.cuda.synchronize()
        assert layer.status() == B.MOE_ERR_DEVICE_TIMEOUT
    finally:
        B.moe_debug_set_wait_limit(0, 0)
    layer.forward(p.X)
    torch.cuda.synchronize()
    assert layer.status() == 0
    idx_o, w_o = p.oracle_routing()
    assert np.array_equal(layer.topk_idx.cpu().numpy(), idx_o)
