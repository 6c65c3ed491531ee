"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test checks the oracle against a brute force, a library routine used as a special
case, a closed form, an invariant of the method, or a number the pages print.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
from expert_routed_ffn_router_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(a):
    return synth.f32_to_bf16_bits(np.asarray(a, np.float32))


def _val(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def _random_router(T, H, E, seed, dup_rows=(), scale=0.3):
    r = np.random.default_rng(seed)
    X = _bits(r.standard_normal((T, H)))
    Wg = r.standard_normal((E, H)) * scale
    for a, b in dup_rows:
        Wg[b] = Wg[a]
    Wg = _bits(Wg)
    bias = r.uniform(-0.1, 0.1, E).astype(np.float32)
    for a, b in dup_rows:
        bias[b] = bias[a]
    return X, Wg, bias


# ---------------------------------------------------------------------------- router
def test_logits_match_library_matmul_and_sigmoid():
    X, Wg, bias = _random_router(7, 96, 12, seed=1)
    _, _, sc = oracle.router(X, Wg, bias, 3, want_scores=True)
    l_ref = _val(X) @ _val(Wg).T                  # numpy float64 GEMM
    np.testing.assert_allclose(sc["logits"], l_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(sc["scores"], expit(l_ref), rtol=1e-14, atol=0)
    np.testing.assert_allclose(sc["sel"], expit(l_ref) + bias.astype(np.float64),
                               rtol=0, atol=1e-15)


def _dominates(sel, a, b):
    return sel[a] > sel[b] or (sel[a] == sel[b] and a < b)


@pytest.mark.parametrize("E,K", [(6, 1), (6, 2), (8, 3), (11, 3), (12, 2)])
def test_topk_bruteforce_all_subsets(E, K):
    X, Wg, bias = _random_router(9, 64, E, seed=E * 10 + K, dup_rows=[(0, E - 1)])
    idx, w, sc = oracle.router(X, Wg, bias, K, want_scores=True)
    for t in range(X.shape[0]):
        sel = sc["sel"][t]
        winners = [S for S in itertools.combinations(range(E), K)
                   if all(_dominates(sel, a, b) for a in S for b in range(E) if b not in S)]
        assert len(winners) == 1
        order = sorted(winners[0], key=lambda e: (-sel[e], e))
        assert list(idx[t]) == order


def test_exact_ties_go_to_lower_index():
    # experts 2 and 5 have identical gate rows and biases: bitwise-equal selection scores
    X, Wg, bias = _random_router(32, 64, 8, seed=3, dup_rows=[(2, 5)])
    idx, _, sc = oracle.router(X, Wg, bias, 4, want_scores=True)
    assert np.array_equal(sc["sel"][:, 2], sc["sel"][:, 5])
    for t in range(32):
        row = list(idx[t])
        if 2 in row and 5 in row:
            assert row.index(2) < row.index(5)
        if 5 in row:
            assert 2 in row


def test_k1_is_argmax_and_kE_is_stable_argsort():
    X, Wg, bias = _random_router(20, 64, 10, seed=4, dup_rows=[(1, 7)])
    i1, w1, sc = oracle.router(X, Wg, bias, 1, want_scores=True)
    assert np.array_equal(i1[:, 0], np.argmax(sc["sel"], axis=1))    # first max on ties
    np.testing.assert_array_equal(w1, 1.0)
    iE, wE = oracle.router(X, Wg, bias, 10)
    assert np.array_equal(iE, np.argsort(-sc["sel"], axis=1, kind="stable"))
    np.testing.assert_allclose(wE.sum(1), 1.0, atol=1e-15)


def test_weights_renormalise_unbiased_scores():
    X, Wg, bias = _random_router(16, 64, 16, seed=5)
    idx, w, sc = oracle.router(X, Wg, bias, 4, want_scores=True)
    s = np.take_along_axis(sc["scores"], idx, axis=1)
    np.testing.assert_allclose(w, s / s.sum(1, keepdims=True), rtol=1e-15)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-15)
    # the bias changes the choice but never the weight formula: a huge bias on one expert
    b2 = bias.copy()
    b2[3] = 10.0
    idx2, w2, sc2 = oracle.router(X, Wg, b2, 4, want_scores=True)
    assert np.all(idx2[:, 0] == 3)
    np.testing.assert_allclose(w2[:, 0], sc2["scores"][:, 3] /
                               np.take_along_axis(sc2["scores"], idx2, 1).sum(1), rtol=1e-15)


# ------------------------------------------------------------------ routing variants
def test_softmax_scores_match_library_softmax():
    X, Wg, bias = _random_router(9, 96, 16, seed=11)
    _, _, sc = oracle.router_ex(X, Wg, bias, 3, scoring="softmax", want_scores=True)
    l_ref = _val(X) @ _val(Wg).T
    s_ref = softmax(l_ref, axis=1)                # scipy, independent of the oracle
    np.testing.assert_allclose(sc["scores"], s_ref, rtol=1e-13, atol=0)
    np.testing.assert_allclose(sc["sel"], s_ref + bias.astype(np.float64), rtol=0, atol=1e-15)


def _group_limited_bruteforce(sel, E, K, n_group, topk_group, group_top):
    """The selection by its definition, every choice found by exhausting the subsets."""
    G = E // n_group
    gscore = [max(sum(sel[e] for e in c)
                  for c in itertools.combinations(range(g * G, (g + 1) * G), group_top))
              for g in range(n_group)]
    dom_g = lambda a, b: gscore[a] > gscore[b] or (gscore[a] == gscore[b] and a < b)
    keep = [S for S in itertools.combinations(range(n_group), topk_group)
            if all(dom_g(a, b) for a in S for b in range(n_group) if b not in S)]
    assert len(keep) == 1
    allowed = [e for e in range(E) if e // G in keep[0]]
    win = [S for S in itertools.combinations(allowed, K)
           if all(_dominates(sel, a, b) for a in S for b in allowed if b not in S)]
    assert len(win) == 1
    return sorted(win[0], key=lambda e: (-sel[e], e))


@pytest.mark.parametrize("scoring", ["sigmoid", "softmax"])
@pytest.mark.parametrize("E,K,n_group,topk_group,group_top", [
    (12, 3, 4, 2, 2), (12, 1, 4, 1, 1), (12, 4, 3, 2, 2), (16, 5, 8, 3, 1), (8, 2, 2, 1, 2)])
def test_group_limited_topk_bruteforce(scoring, E, K, n_group, topk_group, group_top):
    X, Wg, bias = _random_router(12, 64, E, seed=E * 7 + K + n_group, dup_rows=[(0, E - 1)])
    idx, _, sc = oracle.router_ex(X, Wg, bias, K, scoring=scoring, n_group=n_group,
                                  topk_group=topk_group, group_top=group_top, want_scores=True)
    G = E // n_group
    for t in range(X.shape[0]):
        assert list(idx[t]) == _group_limited_bruteforce(sc["sel"][t], E, K, n_group,
                                                         topk_group, group_top)
        assert len({int(e) // G for e in idx[t]}) <= topk_group


def test_one_group_or_every_group_is_the_plain_router():
    X, Wg, bias = _random_router(24, 64, 16, seed=12, dup_rows=[(3, 9)])
    i0, w0 = oracle.router(X, Wg, bias, 4)
    for kw in (dict(n_group=1), dict(n_group=4, topk_group=4, group_top=2),
               dict(n_group=16, topk_group=16)):
        i1, w1 = oracle.router_ex(X, Wg, bias, 4, **kw)
        assert np.array_equal(i0, i1)
        np.testing.assert_array_equal(w0, w1)


def test_equal_group_scores_go_to_lower_group():
    # experts 2,3 (group 1) copy experts 4,5 (group 2): the two groups score the same and
    # a large bias makes them the two best groups; with one group kept, group 1 wins
    X, Wg, bias = _random_router(16, 64, 8, seed=13, dup_rows=[(4, 2), (5, 3)])
    bias[2:6] += 2.0
    idx, _ = oracle.router_ex(X, Wg, bias, 2, n_group=4, topk_group=1, group_top=2)
    assert set(np.unique(idx)) == {2, 3}


def test_mixtral_case_closed_form():
    # softmax scores, one group, renormalised, no bias: the top-K of the logits, weighted
    # by the softmax of the selected logits alone
    X, Wg, _ = _random_router(20, 64, 8, seed=14)
    zero = np.zeros(8, np.float32)
    idx, w = oracle.router_ex(X, Wg, zero, 2, scoring="softmax")
    l_ref = _val(X) @ _val(Wg).T
    assert np.array_equal(idx, np.argsort(-l_ref, axis=1, kind="stable")[:, :2])
    lk = np.take_along_axis(l_ref, idx, 1)
    np.testing.assert_allclose(w, softmax(lk, axis=1), rtol=1e-13)


@pytest.mark.parametrize("scoring", ["sigmoid", "softmax"])
def test_unnormalised_weights_are_the_scores(scoring):
    X, Wg, bias = _random_router(10, 64, 16, seed=15)
    idx, w, sc = oracle.router_ex(X, Wg, bias, 4, scoring=scoring, renorm=False,
                                  n_group=4, topk_group=2, group_top=2, want_scores=True)
    l_ref = _val(X) @ _val(Wg).T
    s_ref = expit(l_ref) if scoring == "sigmoid" else softmax(l_ref, axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(s_ref, idx, 1), rtol=1e-13)


def test_router_ex_rejects_undefined_options():
    X, Wg, bias = _random_router(2, 64, 12, seed=16)
    for kw in (dict(n_group=5), dict(n_group=4, topk_group=5), dict(n_group=4, group_top=4),
               dict(n_group=4, topk_group=1, K=4), dict(n_group=0)):
        K = kw.pop("K", 2)
        with pytest.raises(ValueError):
            oracle.router_ex(X, Wg, bias, K, **kw)


# -------------------------------------------------------------------------- dispatch
def _random_topk(T, E, K, seed):
    r = np.random.default_rng(seed)
    return np.stack([r.permutation(E)[:K] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,K", [(1, 4, 2), (37, 16, 2), (64, 256, 8), (5, 8, 8)])
def test_dispatch_against_stable_argsort(T, E, K):
    idx = _random_topk(T, E, K, seed=T + E)
    d = oracle.dispatch(idx, E)
    flat = idx.ravel()
    order = np.argsort(flat, kind="stable")        # library stable sort of (t, j) by expert
    assert np.array_equal(d["perm"], (order // K).astype(np.int32))
    assert np.array_equal(d["counts"], np.bincount(flat, minlength=E))
    assert np.array_equal(d["offsets"], np.concatenate([[0], np.cumsum(d["counts"])]))
    inv = np.empty_like(order)
    inv[order] = np.arange(T * K)
    assert np.array_equal(d["slot_pos"].ravel(), inv)
    assert d["offsets"][-1] == T * K
    assert sorted(d["perm"].tolist()) == sorted(np.repeat(np.arange(T), K).tolist())


@pytest.mark.parametrize("T,E,K", [(50, 16, 3), (200, 64, 8), (3, 8, 8)])
def test_affinity_is_StS_minus_diag(T, E, K):
    idx = _random_topk(T, E, K, seed=7 * T)
    d = oracle.dispatch(idx, E)
    S = np.zeros((T, E), np.int64)
    S[np.arange(T)[:, None], idx] = 1
    C = S.T @ S - np.diag(d["counts"])
    assert np.array_equal(d["affinity"], C)
    A = d["affinity"]
    assert np.array_equal(A, A.T) and np.all(np.diag(A) == 0)
    assert np.array_equal(A.sum(1), (K - 1) * d["counts"])


def test_pages_worked_examples():
    g = json.load(open(os.path.join(GOLDEN, "pages_worked_examples.json")))
    # 2 tokens x top-8 activate at most 2*8 = 16 experts, each token 8 distinct experts
    b = g["batch_of_two_tokens"]
    X, Wg, bias = _random_router(b["tokens"], 64, g["experts_total"]["value"], seed=11)
    idx, _ = oracle.router(X, Wg, bias, b["topk"])
    d = oracle.dispatch(idx, g["experts_total"]["value"])
    n_act = int((d["counts"] > 0).sum())
    assert n_act <= b["max_active_experts"]
    assert all(len(set(r)) == b["topk"] for r in idx.tolist())
    e = g["avg_active_experts_per_gpu_bs1_ep8"]
    assert e["tokens"] * e["topk"] / e["gpus"] == e["value"]
    assert g["experts_total"]["value"] / 8 == g["experts_per_gpu"]["ep8"]
    assert g["experts_total"]["value"] / 128 == g["experts_per_gpu"]["ep128"]
    # mean tokens per expert m = tokens * k / E: 128 req x q2 x 128 GPUs routed over 256
    m = g["tokens_per_expert_m"]
    T = m["batch_per_gpu"] * m["query_len"] * m["gpus"]
    idx = _random_topk(T, m["experts"], m["topk"], seed=1)
    d = oracle.dispatch(idx, m["experts"], want_affinity=False)
    assert d["counts"].sum() / m["experts"] == m["m"]


# ------------------------------------------------------------------------------- FFN
def test_ffn_scalar_closed_form():
    # H = I = 1: x = 2, W1 = 0.5, W3 = 1.5, W2 = -0.25 -> u = 1, v = 3,
    # h = silu(1) * 3 = 3 * logistic(1), y = -0.75 * logistic(1);
    # logistic(1) = 0.7310585786300049 (e / (1 + e)).
    y = oracle.expert_rows([_bits([2.0])], [_bits([[0.5]])], [_bits([[1.5]])],
                           [_bits([[-0.25]])], 1, 1)
    assert abs(y[0, 0] - (-0.75 * 0.7310585786300049)) < 1e-15


def _tiny_layer(seed, T=11, H=64, E=6, K=2, I=64, Is=64):
    w = synth.Workload("t", T=T, H=H, E=E, K=K, I=I, Is=Is, seed=seed, x_seed=seed)
    return w, synth.host_inputs(w)


def _np_ffn(x, W1, W3, W2):
    u = x @ W1
    v = x @ W3
    return (u * expit(u) * v) @ W2


def test_ffn_matches_library_matmul():
    w, inp = _tiny_layer(2)
    out = oracle.forward(inp)
    X = _val(inp["X"])
    W1, W3, W2 = (_val(inp[n]) for n in ("W1", "W3", "W2"))
    Ysh = _np_ffn(X, _val(inp["W1s"]), _val(inp["W3s"]), _val(inp["W2s"]))
    Y = Ysh.copy()
    for t in range(w.T):
        for j in range(w.K):
            e = out["topk_idx"][t, j]
            Y[t] += out["topk_w"][t, j] * _np_ffn(X[t], W1[e], W3[e], W2[e])
    np.testing.assert_allclose(out["Y"], Y, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("per_pass,shared", [(1, True), (3, True), (16, False)])
def test_expert_by_expert_evaluation_matches_library_matmul(per_pass, shared):
    # layer_tokens_by_expert (the form the DeepSeek-V3-sized parity tests use, fetching a
    # few experts at a time) against numpy float64 matmuls, on a token subset
    w, inp = _tiny_layer(7)
    idx, wts = oracle.router(inp["X"], inp["W_gate"], inp["bias"], w.K)
    X = _val(inp["X"])
    W1, W3, W2 = (_val(inp[n]) for n in ("W1", "W3", "W2"))
    tokens = [w.T - 1, 0, 5, 5, 3]
    fetched = []

    def fetch(e):
        fetched.append(e)
        return inp["W1"][e], inp["W3"][e], inp["W2"][e]
    sh = (inp["W1s"], inp["W3s"], inp["W2s"]) if shared else None
    Y = oracle.layer_tokens_by_expert(inp["X"], idx, wts, fetch, sh, tokens, w.I, w.Is,
                                      experts_per_pass=per_pass)
    used = sorted({int(e) for t in tokens for e in idx[t]})
    assert fetched == used                      # every needed expert once, in order
    for q, t in enumerate(tokens):
        ref = _np_ffn(X[t], _val(inp["W1s"]), _val(inp["W3s"]), _val(inp["W2s"])) if shared \
            else np.zeros(w.H)
        for j in range(w.K):
            e = idx[t, j]
            ref = ref + wts[t, j] * _np_ffn(X[t], W1[e], W3[e], W2[e])
        np.testing.assert_allclose(Y[q], ref, rtol=1e-12, atol=1e-13)


def test_identical_experts_collapse():
    w, inp = _tiny_layer(3)
    for n in ("W1", "W3", "W2"):
        inp[n][:] = inp[n][0]
    out = oracle.forward(inp)
    X = _val(inp["X"])
    ffn = _np_ffn(X, _val(inp["W1"][0]), _val(inp["W3"][0]), _val(inp["W2"][0]))
    sh = _np_ffn(X, _val(inp["W1s"]), _val(inp["W3s"]), _val(inp["W2s"]))
    # sum_j w_j FFN(x) = FFN(x) because the weights sum to one
    np.testing.assert_allclose(out["Y"], ffn + sh, rtol=1e-12, atol=1e-13)


def test_zero_up_projection_leaves_shared_expert_only():
    w, inp = _tiny_layer(4)
    inp["W3"][:] = 0
    out = oracle.forward(inp)
    X = _val(inp["X"])
    sh = _np_ffn(X, _val(inp["W1s"]), _val(inp["W3s"]), _val(inp["W2s"]))
    np.testing.assert_allclose(out["Y"], sh, rtol=1e-12, atol=1e-14)


def test_linear_in_down_projection_and_no_shared():
    w, inp = _tiny_layer(5, Is=0)
    inp["W1s"] = inp["W3s"] = inp["W2s"] = None
    y1 = oracle.forward(inp)["Y"]
    inp2 = dict(inp)
    inp2["W2"] = _bits(_val(inp["W2"]) * 2.0)      # doubling is exact in bf16
    y2 = oracle.forward(inp2)["Y"]
    np.testing.assert_allclose(y2, 2.0 * y1, rtol=1e-14, atol=1e-15)


def test_k1_no_shared_is_the_selected_expert():
    w, inp = _tiny_layer(6, K=1, Is=0)
    inp["W1s"] = inp["W3s"] = inp["W2s"] = None
    out = oracle.forward(inp)
    X = _val(inp["X"])
    for t in range(w.T):
        e = out["topk_idx"][t, 0]
        ref = _np_ffn(X[t], _val(inp["W1"][e]), _val(inp["W3"][e]), _val(inp["W2"][e]))
        np.testing.assert_allclose(out["Y"][t], ref, rtol=1e-12, atol=1e-14)


def test_bf16_encoding_round_to_nearest_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> ties to even (1.0);
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6 -> even is 1 + 2^-6
    v = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.5, 0.0, 3e-30], np.float32)
    b = synth.f32_to_bf16_bits(v)
    assert b[0] == 0x3F80 and b[1] == 0x3F82 and b[2] == 0xC020 and b[3] == 0
    np.testing.assert_array_equal(_val(b)[:4], [1.0, 1 + 2 ** -6, -2.5, 0.0])
    assert math.isclose(_val(b)[4], 3e-30, rel_tol=2 ** -8)


def test_combine_one_hot_and_linearity():
    r = np.random.default_rng(9)
    T, K, H = 6, 3, 32
    Yp = _bits(r.standard_normal((T * K, H)))
    slot = r.permutation(T * K).reshape(T, K).astype(np.int32)
    onehot = np.zeros((T, K))
    onehot[:, 1] = 1.0
    Y = oracle.combine(Yp, slot, onehot)
    np.testing.assert_array_equal(Y, _val(Yp)[slot[:, 1]])       # picks one row exactly
    w = r.uniform(0, 1, (T, K))
    sh = r.standard_normal((T, H))
    Y1 = oracle.combine(Yp, slot, w, sh)
    ref = np.einsum("tk,tkh->th", w, _val(Yp)[slot]) + sh      # library contraction
    np.testing.assert_allclose(Y1, ref, rtol=1e-14, atol=1e-14)
