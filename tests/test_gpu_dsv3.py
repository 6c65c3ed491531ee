"""GPU parity at the DeepSeek-V3 shape (H=7168, E=256, K=8, I=I_shared=2048) in the launch
configuration the benchmark times: routing, counts and affinity bit-exact over every token,
Y on sampled tokens that the oracle evaluates one by one."""
import numpy as np
import pytest

from expert_routed_ffn_router_gb300 import synth

from gpu_common import DEV, Problem, check_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsv3_weights():
    w = synth.workload("decode")
    return synth.expert_weights_device(w, DEV)


def _sample(T, n):
    return sorted({0, T - 1, *np.linspace(0, T - 1, n).astype(int).tolist()})


def test_decode_T128(dsv3_weights):
    w = synth.workload("decode")
    check_layer(Problem(w, weights_dev=dsv3_weights), tokens=_sample(w.T, 4))


@pytest.mark.parametrize("T", [2, 8, 64])
def test_batch_sweep(dsv3_weights, T):
    w = synth.workload(f"sweep{T}")
    r = check_layer(Problem(w, weights_dev=dsv3_weights),
                    tokens=None if T <= 2 else _sample(T, 3))
    n_act = int((r["disp"]["counts"] > 0).sum())
    assert n_act <= min(w.E, T * w.K)


def test_prefill_T16384(dsv3_weights):
    w = synth.workload("prefill")
    check_layer(Problem(w, weights_dev=dsv3_weights), tokens=_sample(w.T, 2))


def test_skewed_T8192(dsv3_weights):
    w = synth.workload("skewed")
    r = check_layer(Problem(w, weights_dev=dsv3_weights), tokens=_sample(w.T, 2))
    assert r["disp"]["counts"].max() >= 0.95 * w.T  # the most popular experts: nearly every token


def test_dispatch_gathers_token_by_token_at_prefill_size():
    # X of 16384 x 7168 bf16 (235 MB) is larger than half of L2: the row gather then runs
    # token by token (each token row read once, written to its K slots)
    import torch
    from expert_routed_ffn_router_gb300 import binding as B

    w = synth.workload("prefill")
    r = synth.routing_inputs(w)
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(DEV)
    X, Wg, bias = to(r["X"]), to(r["W_gate"]), torch.from_numpy(r["bias"]).to(DEV)
    T, H, E, K = w.T, w.H, w.E, w.K
    ws = torch.zeros(B.moe_workspace_bytes(T, H, E, K, w.I, w.Is), dtype=torch.uint8, device=DEV)
    idx = torch.empty(T, K, dtype=torch.int32, device=DEV)
    wt = torch.empty(T, K, dtype=torch.float32, device=DEV)
    B.moe_router_topk(X, Wg, bias, K, idx, wt, ws)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * K, dtype=torch.int32, device=DEV)
    slot = torch.empty(T, K, dtype=torch.int32, device=DEV)
    Xp = torch.empty(T * K, H, dtype=torch.bfloat16, device=DEV)
    B.moe_dispatch(X, idx, E, counts, offsets, perm, slot, Xp, None, ws)
    torch.cuda.synchronize()
    assert B.moe_read_status(ws) == 0
    p = perm.long()
    assert torch.equal(Xp.view(torch.int16), X.view(torch.int16)[p])
    # slot_pos is the inverse of perm, and perm lists every (token, slot) once
    tok = torch.arange(T, device=DEV).unsqueeze(1).expand(T, K)
    assert torch.equal(p[slot.long()], tok)
