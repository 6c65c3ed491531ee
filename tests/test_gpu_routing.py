"""Routing options of other MoE families on the GPU against the oracle ("Lower latency and
higher throughput with multi-node DeepSeek deployment", MoE Router: one router serves every
MoE model; DeepSeek routing selects among expert groups, Mixtral's is the one-group case).
Softmax scoring, group-limited top-k and unnormalised weights: indices bit-exact, weights
within 1e-5, in every router launch configuration (one-warp-per-expert GEMV for T <= 4,
fused GEMM + finalise up to 4096 tokens, GEMM + one-warp-per-token finalise beyond)."""
import numpy as np
import pytest
import torch

import oracle
from expert_routed_ffn_router_gb300 import binding as B
from expert_routed_ffn_router_gb300 import synth

from gpu_common import DEV, W_MAX_ABS, Problem, check_layer, host_to_device_bf16

pytestmark = pytest.mark.gpu

OPTS = {
    # DeepSeek-V3-like: sigmoid, 8 groups of 32, the 4 best groups by their top-2 sum
    "groups_top2": dict(scoring="sigmoid", n_group=8, topk_group=4, group_top=2),
    # DeepSeek-V2-like: softmax, groups scored by their best expert, weights not renormalised
    "softmax_groups_max": dict(scoring="softmax", n_group=8, topk_group=3, group_top=1,
                               renorm=False),
    # Mixtral-like: softmax over all experts, renormalised over the selected ones
    "softmax": dict(scoring="softmax"),
    "sigmoid_unnormalised": dict(renorm=False),
}


def _run_router(r, K, opts):
    T = r["X"].shape[0]
    E, H = r["W_gate"].shape
    X = host_to_device_bf16(r["X"])
    Wg = host_to_device_bf16(r["W_gate"])
    bias = torch.from_numpy(r["bias"]).to(DEV)
    ws = torch.zeros(B.moe_workspace_bytes(T, H, E, K, 64, 0), dtype=torch.uint8, device=DEV)
    idx = torch.empty(T, K, dtype=torch.int32, device=DEV)
    wt = torch.empty(T, K, dtype=torch.float32, device=DEV)
    B.moe_router_topk_ex(X, Wg, bias, K, opts, idx, wt, ws)
    torch.cuda.synchronize()
    assert B.moe_read_status(ws) == 0
    return idx.cpu().numpy(), wt.cpu().numpy().astype(np.float64)


def _check_router(r, K, opts):
    idx_g, w_g = _run_router(r, K, opts)
    idx_o, w_o = oracle.router_ex(r["X"], r["W_gate"], r["bias"], K, **opts)
    bad = np.nonzero((idx_g != idx_o).any(1))[0]
    assert bad.size == 0, f"tokens {bad[:8]}: gpu {idx_g[bad[:2]]} oracle {idx_o[bad[:2]]}"
    assert np.abs(w_g - w_o).max() <= W_MAX_ABS
    return idx_o, w_o


@pytest.mark.parametrize("name", sorted(OPTS))
@pytest.mark.parametrize("T", [1, 3, 7, 200, 4100])
def test_router_options_dsv3_shape(name, T):
    w = synth.workload("decode", T=T, x_seed=T + 11)
    _check_router(synth.routing_inputs(w), w.K, OPTS[name])


@pytest.mark.parametrize("name", sorted(OPTS))
def test_router_options_exact_and_near_ties(name):
    # gate rows copied across and inside groups (exact ties: lower index / lower group
    # first) and rows one bf16 ulp apart (near ties: only the re-scored path decides)
    w = synth.workload("decode", T=96, x_seed=5)
    r = synth.routing_inputs(w)
    for a, b in ((3, 40), (7, 8), (100, 230), (64, 65)):
        r["W_gate"][b] = r["W_gate"][a]
        r["bias"][b] = r["bias"][a]
    for a, b in ((12, 13), (150, 190)):
        r["W_gate"][b] = r["W_gate"][a]
        r["W_gate"][b, 99] = r["W_gate"][a, 99] + 1
        r["bias"][b] = r["bias"][a]
    r["bias"][[3, 40, 7, 8]] += 0.5        # make the tied experts win often
    idx, _ = _check_router(r, w.K, OPTS[name])
    both = [row for row in idx.tolist() if 3 in row and 40 in row]
    assert all(row.index(3) < row.index(40) for row in both)


def test_groups_tie_on_score_lower_group_wins():
    # groups 1 and 5 hold identical gate rows and biases: equal group scores every token
    w = synth.workload("decode", T=64, x_seed=9)
    r = synth.routing_inputs(w)
    r["W_gate"][160:192] = r["W_gate"][32:64]
    r["bias"][160:192] = r["bias"][32:64]
    r["bias"][32:64] += 0.3
    r["bias"][160:192] += 0.3
    opts = dict(scoring="sigmoid", n_group=8, topk_group=1, group_top=2)
    idx, _ = _check_router(r, w.K, opts)
    assert np.all((idx >= 32) & (idx < 64))


@pytest.mark.parametrize("topk_group", [1, 2, 4])
def test_groups_near_tie_is_decided_exactly(topk_group):
    # group 5 copies group 1 with one bf16 ulp added to one element of every row: the two
    # group scores differ far inside the fp32 bound, so the group choice is left to the
    # re-scored candidates
    w = synth.workload("decode", T=80, x_seed=10)
    r = synth.routing_inputs(w)
    r["W_gate"][160:192] = r["W_gate"][32:64]
    r["W_gate"][160:192, 7] += 1
    r["bias"][160:192] = r["bias"][32:64]
    r["bias"][32:64] += 0.3
    r["bias"][160:192] += 0.3
    for group_top in (1, 2):
        opts = dict(scoring="sigmoid", n_group=8, topk_group=topk_group, group_top=group_top)
        _check_router(r, w.K, opts)


@pytest.mark.parametrize("name", ["groups_top2", "softmax_groups_max"])
def test_layer_forward_with_routing_options(name):
    w = synth.Workload("rt", T=150, H=256, E=32, K=4, I=128, Is=128, seed=21, x_seed=22)
    opts = dict(OPTS[name], n_group=4, topk_group=2)
    check_layer(Problem(w, opts=opts))


@pytest.mark.parametrize("opts", [{}, OPTS["groups_top2"]])
def test_large_batch_tiles_with_ragged_edges(opts):
    # the 128-token x 64-expert tile GEMM of batches above 4096 tokens: a partial last
    # token tile (4300 = 33 x 128 + 76), a partial last expert tile (72 = 64 + 8) and a
    # K split that does not divide the 15 stages of H = 960
    w = synth.Workload("large_ragged", T=4300, H=960, E=72 if not opts else 64, K=6,
                       I=64, Is=0, seed=21, x_seed=22)
    _check_router(synth.routing_inputs(w), w.K, opts)


@pytest.mark.parametrize("opts", [{}, OPTS["groups_top2"]])
@pytest.mark.parametrize("T", [5, 40, 4200])
def test_non_finite_scores_still_give_valid_indices(opts, T):
    # rows of X with a NaN, an infinity, or magnitudes whose fp32 products overflow: the
    # exact top-k is undefined there, but the router must still write K distinct in-range
    # experts per token (the certified selection falls back to re-scoring every expert)
    w = synth.workload("decode", T=T, x_seed=T + 17)
    r = synth.routing_inputs(w)
    big = synth.f32_to_bf16_bits(np.full(w.H, 3.0e38, dtype=np.float32))
    r["X"][0, 5] = synth.f32_to_bf16_bits(np.array([np.nan], dtype=np.float32))[0]
    r["X"][1, 7] = synth.f32_to_bf16_bits(np.array([np.inf], dtype=np.float32))[0]
    r["X"][T - 1] = big
    idx, wt = _run_router(r, w.K, opts)
    assert idx.min() >= 0 and idx.max() < w.E
    assert all(len(set(row)) == w.K for row in idx.tolist())
    # the finite rows are unaffected
    ok = np.ones(T, bool)
    ok[[0, 1, T - 1]] = False
    idx_o, w_o = oracle.router_ex(r["X"][ok], r["W_gate"], r["bias"], w.K, **opts)
    assert np.array_equal(idx[ok], idx_o)
