"""Expert indices outside [0, E) given to moe_dispatch: the call records MOE_ERR_INVALID_ARG in
the workspace's status word, the rejected pairs get no row (slot_pos = -1; counts, perm, Xp
and affinity hold the valid pairs only) and nothing is written out of bounds -- on the
one-launch dispatch (45 tokens), the multi-launch one gathering row by row (300 tokens) and
token by token (5000 tokens of 7168 features).  moe_combine skips the rejected slots.  The
debug mode (moe_debug_set_sync_status) returns the status word from the call itself, for
the dispatch and for a layer whose bounded waits run out."""
import numpy as np
import pytest
import torch

from expert_routed_ffn_router_gb300 import binding as B
from expert_routed_ffn_router_gb300 import synth

from gpu_common import DEV, Problem, host_to_device_bf16

pytestmark = pytest.mark.gpu

MOE_ERR_INVALID_ARG = -1


def _routing_with_bad_indices(T, E, K, seed=11):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, size=K, replace=False) for _ in range(T)]).astype(np.int32)
    for t, j, v in ((0, 0, E), (T // 2, K - 1, -3), (T - 1, 1 % K, E + 1000)):
        idx[t, j] = v
    return idx


def _dispatch(w, idx):
    T, H, E, K = w.T, w.H, w.E, w.K
    r = synth.routing_inputs(w)
    X = host_to_device_bf16(r["X"])
    ws = torch.zeros(B.moe_workspace_bytes(T, H, E, K, w.I, w.Is), dtype=torch.uint8, device=DEV)
    out = dict(counts=torch.empty(E, dtype=torch.int32, device=DEV),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=DEV),
               perm=torch.full((T * K,), -7, dtype=torch.int32, device=DEV),
               slot=torch.full((T, K), -7, dtype=torch.int32, device=DEV),
               Xp=torch.zeros(T * K, H, dtype=torch.bfloat16, device=DEV),
               aff=torch.empty(E, E, dtype=torch.int32, device=DEV))
    B.moe_dispatch(X, torch.from_numpy(idx).to(DEV), E, out["counts"], out["offsets"],
                   out["perm"], out["slot"], out["Xp"], out["aff"], ws)
    return r, X, ws, out


@pytest.mark.parametrize("name,T", [("tiny", 45), ("tiny", 300), ("decode", 5000)])
def test_out_of_range_experts_are_rejected_and_get_no_row(name, T):
    w = synth.workload(name, T=T)
    E, K = w.E, w.K
    idx = _routing_with_bad_indices(T, E, K)
    r, X, ws, o = _dispatch(w, idx)
    assert B.moe_read_status(ws) == MOE_ERR_INVALID_ARG
    valid = (idx >= 0) & (idx < E)
    counts = np.bincount(idx[valid], minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    assert np.array_equal(o["counts"].cpu().numpy(), counts)
    assert np.array_equal(o["offsets"].cpu().numpy(), offsets)
    n = int(offsets[-1])
    assert n == T * K - 3
    slot = o["slot"].cpu().numpy()
    perm = o["perm"].cpu().numpy()
    assert np.all(slot[~valid] == -1)
    # the valid pairs: rows ordered by (expert, token), slot_pos their inverse
    for e in range(E):
        toks = np.nonzero((idx == e).any(axis=1))[0]
        assert np.array_equal(perm[offsets[e]:offsets[e + 1]], toks)
    ts, js = np.nonzero(valid)
    assert np.array_equal(perm[slot[ts, js]], ts)
    assert np.all(perm[n:] == -7)                    # rows past the valid ones untouched
    Xp = o["Xp"].view(torch.int16).cpu().numpy()
    assert np.array_equal(Xp[:n], r["X"].view(np.int16)[perm[:n]])
    assert not Xp[n:].any()                          # nothing gathered past them
    S = np.zeros((T, E), np.int64)
    S[ts, idx[ts, js]] = 1
    A = S.T @ S
    np.fill_diagonal(A, 0)
    assert np.array_equal(o["aff"].cpu().numpy(), A)

    # combine over the dispatch's slots: the rejected ones contribute nothing
    rng = np.random.default_rng(5)
    Yp_h = synth.f32_to_bf16_bits(rng.standard_normal((T * K, w.H)).astype(np.float32))
    wt = rng.random((T, K)).astype(np.float32)
    Y = torch.empty(T, w.H, dtype=torch.float32, device=DEV)
    B.moe_combine(host_to_device_bf16(Yp_h), o["slot"], torch.from_numpy(wt).to(DEV), None, Y)
    Yp64 = synth.bf16_bits_to_f32(Yp_h).astype(np.float64)
    Y_ref = np.zeros((T, w.H))
    for j in range(K):
        m = valid[:, j]
        Y_ref[m] += wt[m, j, None].astype(np.float64) * Yp64[slot[m, j]]
    assert np.abs(Y.cpu().numpy() - Y_ref).max() <= 1e-4


def test_debug_mode_returns_the_status_word_from_the_call():
    w = synth.workload("tiny", T=45)
    idx = _routing_with_bad_indices(w.T, w.E, w.K)
    B.moe_debug_set_sync_status(True)
    try:
        with pytest.raises(B.MoeError) as ei:
            _dispatch(w, idx)
        assert ei.value.status == MOE_ERR_INVALID_ARG
        # a layer whose bounded waits run out: the forward call itself reports it
        p = Problem(w)
        layer = B.MoELayer(p.dev, w.T, w.K)
        B.moe_debug_set_wait_limit(50_000_000, inject_stall=1)   # 50 ms
        try:
            with pytest.raises(B.MoeError) as ei:
                layer.forward(p.X)
            assert ei.value.status == B.MOE_ERR_DEVICE_TIMEOUT
        finally:
            B.moe_debug_set_wait_limit(0, 0)
        layer.forward(p.X)                               # a clean call returns MOE_OK
    finally:
        B.moe_debug_set_sync_status(False)
    torch.cuda.synchronize()
    assert layer.status() == 0


@pytest.mark.parametrize("bad", ["decreasing", "past_rows", "negative"])
def test_expert_ffn_rejects_offsets_outside_its_rows(bad):
    # moe_expert_ffn reads the group offsets on the device only: offsets that are not
    # non-decreasing within [0, rows] make the launch record MOE_ERR_INVALID_ARG and run no
    # tile (nothing written), and the next valid call on the same buffers runs normally
    w = synth.workload("tiny", T=40)
    p = Problem(w)
    T, H, E, K, I = w.T, w.H, w.E, w.K, w.I
    rows = T * K
    good = np.linspace(0, rows, E + 1).astype(np.int32)
    off = good.copy()
    if bad == "decreasing":
        off[3], off[4] = good[4], good[3]
    elif bad == "past_rows":
        off[-1] = rows + 64
    else:
        off[0] = -16
    rng = np.random.default_rng(2)
    Xp = host_to_device_bf16(synth.f32_to_bf16_bits(rng.standard_normal((rows, H)).astype(np.float32)))
    Yp = torch.full((rows, H), 7.0, dtype=torch.float32, device=DEV)
    ws = torch.zeros(B.moe_expert_ffn_workspace_bytes(rows, E, I), dtype=torch.uint8, device=DEV)
    B.moe_expert_ffn(Xp, torch.from_numpy(off).to(DEV), E, p.dev["W1"], p.dev["W3"], p.dev["W2"],
                     Yp, ws)
    assert B.moe_read_status(ws) == MOE_ERR_INVALID_ARG
    assert bool(torch.all(Yp == 7.0))
    B.moe_expert_ffn(Xp, torch.from_numpy(good).to(DEV), E, p.dev["W1"], p.dev["W3"],
                     p.dev["W2"], Yp, ws)
    assert B.moe_read_status(ws) == 0
    assert not bool(torch.any(Yp == 7.0))


def test_combine_skips_rows_outside_its_inputs():
    # slot_pos entries outside [0, T*K) (here past the end and far past it) contribute
    # nothing; the other slots are summed as usual
    T, H, K = 45, 256, 2
    rng = np.random.default_rng(8)
    slot = rng.permutation(T * K).astype(np.int32).reshape(T, K)
    slot[3, 0], slot[17, 1], slot[44, 0] = T * K + 5, 1 << 30, -2
    keep = (slot >= 0) & (slot < T * K)
    Yp_h = synth.f32_to_bf16_bits(rng.standard_normal((T * K, H)).astype(np.float32))
    wt = rng.random((T, K)).astype(np.float32)
    Y = torch.empty(T, H, dtype=torch.float32, device=DEV)
    B.moe_combine(host_to_device_bf16(Yp_h), torch.from_numpy(slot).to(DEV),
                  torch.from_numpy(wt).to(DEV), None, Y)
    Yp64 = synth.bf16_bits_to_f32(Yp_h).astype(np.float64)
    Y_ref = np.zeros((T, H))
    for j in range(K):
        m = keep[:, j]
        Y_ref[m] += wt[m, j, None].astype(np.float64) * Yp64[slot[m, j]]
    assert np.abs(Y.cpu().numpy() - Y_ref).max() <= 1e-4
