"""ctypes front end of the fp64 CPU oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's
CPU-baseline leg may import this module; the product path never does.  It shares no code
with the CUDA library.

Inputs are numpy arrays: bf16 values travel as ``uint16`` bit patterns, the bias as
``float32``.  Every function returns freshly allocated numpy arrays.

Page citations (by title and section):
  * "Lower latency and higher throughput with multi-node DeepSeek deployment":
    Expert Parallelism (routed + shared experts, weighted sum), MoE Router (index-tracking
    sort, per-expert aggregated routing info), Quantization (SiLU activation).
  * "DeepSeek-V4.1-Flash" (vLLM), Kernels / Mega-Gate (gate GEMM, scoring, bias, top-k).
  * "GRACE-MoE", Core Idea 1 (expert affinity matrix A).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libmoe_oracle.so")
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/libmoe_oracle.so (gcc, OpenMP, -O2)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_oracle())
        P = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_router.argtypes = [P, P, P, i, i, i, i, P, P, P, P, P]
        lib.oracle_router.restype = i
        lib.oracle_router_ex.argtypes = [P, P, P, i, i, i, i, i, i, i, i, i, P, P, P, P, P]
        lib.oracle_router_ex.restype = i
        lib.oracle_dispatch.argtypes = [P, i, i, i, P, P, P, P, P]
        lib.oracle_dispatch.restype = i
        lib.oracle_expert_rows.argtypes = [P, P, P, P, i, i, i, P]
        lib.oracle_expert_rows.restype = i
        lib.oracle_layer_tokens.argtypes = [P, i, i, i, i, P, P, P, P, P, P, P, P, P, i, P]
        lib.oracle_layer_tokens.restype = i
        lib.oracle_combine.argtypes = [P, P, P, P, i, i, i, P]
        lib.oracle_combine.restype = i
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i
        lib.oracle_set_num_threads.argtypes = [i]
        lib.oracle_set_num_threads.restype = i
        _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 inputs travel as uint16 bit patterns, got {a.dtype}")
    return a


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> int:
    """Threads for this thread's later oracle calls; returns the previous count."""
    return int(_load().oracle_set_num_threads(int(n)))


def router(X: np.ndarray, W_gate: np.ndarray, bias: np.ndarray, K: int,
           want_scores: bool = False):
    """Gate GEMM -> sigmoid -> + bias -> top-K -> renormalised weights (fp64).

    Returns (topk_idx int32 [T,K], topk_w float64 [T,K]) and, with want_scores,
    a dict of the [T,E] logits, sigmoid scores and biased selection scores."""
    X = _u16(X)
    W_gate = _u16(W_gate)
    bias = np.ascontiguousarray(bias, dtype=np.float32)
    T, H = X.shape
    E = W_gate.shape[0]
    assert W_gate.shape == (E, H) and bias.shape == (E,)
    idx = np.zeros((T, K), np.int32)
    w = np.zeros((T, K), np.float64)
    extra = {}
    if want_scores:
        extra = {n: np.zeros((T, E), np.float64) for n in ("logits", "scores", "sel")}
    rc = _load().oracle_router(_p(X), _p(W_gate), _p(bias), T, H, E, K, _p(idx), _p(w),
                               _p(extra.get("logits")), _p(extra.get("scores")),
                               _p(extra.get("sel")))
    if rc != 0:
        raise ValueError(f"oracle_router rejected its arguments ({rc})")
    return (idx, w, extra) if want_scores else (idx, w)


SCORING = {"sigmoid": 0, "softmax": 1}


def router_ex(X: np.ndarray, W_gate: np.ndarray, bias: np.ndarray, K: int,
              scoring: str = "sigmoid", n_group: int = 1, topk_group: int = 1,
              group_top: int = 1, renorm: bool = True, want_scores: bool = False):
    """Router with the options of other MoE families (fp64).

    scoring: "sigmoid" or "softmax" (over the token's E logits); the E experts form
    n_group groups of E/n_group consecutive experts, a group scores the sum of its
    group_top largest sel = s + bias, and the top-K is taken inside the topk_group best
    groups; renorm divides the selected s by their sum (else the weights are s)."""
    X = _u16(X)
    W_gate = _u16(W_gate)
    bias = np.ascontiguousarray(bias, dtype=np.float32)
    T, H = X.shape
    E = W_gate.shape[0]
    assert W_gate.shape == (E, H) and bias.shape == (E,)
    idx = np.zeros((T, K), np.int32)
    w = np.zeros((T, K), np.float64)
    extra = {}
    if want_scores:
        extra = {n: np.zeros((T, E), np.float64) for n in ("logits", "scores", "sel")}
    rc = _load().oracle_router_ex(_p(X), _p(W_gate), _p(bias), T, H, E, K, SCORING[scoring],
                                  n_group, topk_group, group_top, int(bool(renorm)),
                                  _p(idx), _p(w), _p(extra.get("logits")),
                                  _p(extra.get("scores")), _p(extra.get("sel")))
    if rc != 0:
        raise ValueError(f"oracle_router_ex rejected its arguments ({rc})")
    return (idx, w, extra) if want_scores else (idx, w)


def dispatch(topk_idx: np.ndarray, E: int, want_affinity: bool = True):
    """Counts, offsets, stable permutation (expert, token), slot positions, affinity."""
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, K = topk_idx.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * K, np.int32)
    slot_pos = np.zeros((T, K), np.int32)
    aff = np.zeros((E, E), np.int32) if want_affinity else None
    rc = _load().oracle_dispatch(_p(topk_idx), T, E, K, _p(counts), _p(offsets), _p(perm),
                                 _p(slot_pos), _p(aff))
    if rc != 0:
        raise ValueError(f"oracle_dispatch rejected its arguments ({rc})")
    return dict(counts=counts, offsets=offsets, perm=perm, slot_pos=slot_pos, affinity=aff)


def expert_rows(xrows, W1s, W3s, W2s, H: int, I: int) -> np.ndarray:
    """y[n] = (silu(x_n W1_n) * (x_n W3_n)) W2_n for lists of per-row bf16 arrays."""
    n = len(xrows)
    keep = [_u16(a) for a in list(xrows) + list(W1s) + list(W3s) + list(W2s)]
    PtrArr = ctypes.c_void_p * max(n, 1)
    arrs = [PtrArr(*[a.ctypes.data for a in keep[g * n:(g + 1) * n]]) for g in range(4)]
    y = np.zeros((n, H), np.float64)
    rc = _load().oracle_expert_rows(*[ctypes.cast(a, ctypes.c_void_p) for a in arrs],
                                    n, H, I, _p(y))
    if rc != 0:
        raise ValueError(f"oracle_expert_rows rejected its arguments ({rc})")
    del keep
    return y


def layer_tokens(X: np.ndarray, topk_idx: np.ndarray, topk_w: np.ndarray,
                 W1: dict, W3: dict, W2: dict, W1s, W3s, W2s, tokens, I: int,
                 Is: int) -> np.ndarray:
    """Y[q] = sum_j w[t,j] FFN_{e_tj}(X[t]) + FFN_shared(X[t]) for t = tokens[q] (fp64).

    W1/W3/W2 map an expert index to its bf16 [H,I] / [H,I] / [I,H] arrays (only the
    experts the listed tokens use need to be present)."""
    X = _u16(X)
    T, H = X.shape
    K = topk_idx.shape[1]
    E = max(int(topk_idx.max()) + 1, max(W1.keys()) + 1 if W1 else 1)
    keep = []
    tabs = []
    for d in (W1, W3, W2):
        arr = (ctypes.c_void_p * E)()
        for e, a in d.items():
            a = _u16(a)
            keep.append(a)
            arr[e] = a.ctypes.data
        tabs.append(arr)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    topk_w = np.ascontiguousarray(topk_w, dtype=np.float64)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    sh = [None if a is None else _u16(a) for a in (W1s, W3s, W2s)]
    Y = np.zeros((len(tokens), H), np.float64)
    rc = _load().oracle_layer_tokens(_p(X), H, I, Is, K, _p(topk_idx), _p(topk_w),
                                     *[ctypes.cast(a, ctypes.c_void_p) for a in tabs],
                                     _p(sh[0]), _p(sh[1]), _p(sh[2]),
                                     _p(tokens), len(tokens), _p(Y))
    if rc != 0:
        raise ValueError(f"oracle_layer_tokens rejected its arguments ({rc})")
    del keep
    return Y


def layer_tokens_by_expert(X: np.ndarray, topk_idx: np.ndarray, topk_w: np.ndarray,
                           fetch_expert, shared, tokens, I: int, Is: int,
                           experts_per_pass: int = 16) -> np.ndarray:
    """The same Y as ``layer_tokens`` (fp64), evaluated expert by expert so that only a few
    experts' weights need to be on the host at a time.

    fetch_expert(e) returns the bf16 (W1 [H,I], W3 [H,I], W2 [I,H]) arrays of expert e;
    shared is (W1s, W3s, W2s) or None.  The (token, slot) pairs of the listed tokens are
    grouped by expert; each pass fetches `experts_per_pass` experts and evaluates all their
    pairs (``expert_rows``).  Then Y[q] = sum_j w[t,j] y[q,j] + y_shared[q], j ascending,
    for t = tokens[q]."""
    X = _u16(X)
    H = X.shape[1]
    K = topk_idx.shape[1]
    tokens = np.asarray(tokens, dtype=np.int64)
    n = len(tokens)
    ysel = np.zeros((n, K, H), np.float64)
    pairs = {}
    for q, t in enumerate(tokens):
        for j in range(K):
            pairs.setdefault(int(topk_idx[t, j]), []).append((q, j))
    experts = sorted(pairs)
    for c in range(0, len(experts), experts_per_pass):
        chunk = experts[c:c + experts_per_pass]
        weights = {e: fetch_expert(e) for e in chunk}
        rows = [(e, q, j) for e in chunk for (q, j) in pairs[e]]
        y = expert_rows([X[tokens[q]] for (_, q, _) in rows],
                        [weights[e][0] for (e, _, _) in rows],
                        [weights[e][1] for (e, _, _) in rows],
                        [weights[e][2] for (e, _, _) in rows], H, I)
        for r, (_, q, j) in enumerate(rows):
            ysel[q, j] = y[r]
        del weights
    Y = np.zeros((n, H), np.float64)
    for j in range(K):
        Y += topk_w[tokens, j][:, None] * ysel[:, j]
    if shared is not None and Is > 0:
        W1s, W3s, W2s = shared
        Y += expert_rows([X[t] for t in tokens], [W1s] * n, [W3s] * n, [W2s] * n, H, Is)
    return Y


def combine(Yp: np.ndarray, slot_pos: np.ndarray, topk_w: np.ndarray,
            Ysh: np.ndarray | None = None) -> np.ndarray:
    """Y[t] = sum_j topk_w[t,j] * Yp[slot_pos[t,j]] (+ Ysh[t]); Yp bf16 bits [rows,H]."""
    Yp = _u16(Yp)
    slot_pos = np.ascontiguousarray(slot_pos, dtype=np.int32)
    topk_w = np.ascontiguousarray(topk_w, dtype=np.float64)
    T, K = slot_pos.shape
    H = Yp.shape[1]
    if Ysh is not None:
        Ysh = np.ascontiguousarray(Ysh, dtype=np.float64)
    Y = np.zeros((T, H), np.float64)
    rc = _load().oracle_combine(_p(Yp), _p(slot_pos), _p(topk_w), _p(Ysh), T, H, K, _p(Y))
    if rc != 0:
        raise ValueError(f"oracle_combine rejected its arguments ({rc})")
    return Y


def forward(inp: dict) -> dict:
    """The whole layer for every token of a small problem held in host numpy arrays.

    ``inp`` holds X, W_gate, bias, W1, W3, W2 ([E,...] uint16), W1s, W3s, W2s (or None),
    K and optionally ``routing`` (keyword options of router_ex).  Returns the routing,
    dispatch bookkeeping and Y (float64 [T,H])."""
    X, K = inp["X"], int(inp["K"])
    T, H = X.shape
    E, _, I = inp["W1"].shape
    Is = 0 if inp.get("W1s") is None else inp["W1s"].shape[1]
    routing = inp.get("routing")
    if routing:
        idx, w = router_ex(X, inp["W_gate"], inp["bias"], K, **routing)
    else:
        idx, w = router(X, inp["W_gate"], inp["bias"], K)
    d = dispatch(idx, E)
    W1 = {e: inp["W1"][e] for e in range(E)}
    W3 = {e: inp["W3"][e] for e in range(E)}
    W2 = {e: inp["W2"][e] for e in range(E)}
    Y = layer_tokens(X, idx, w, W1, W3, W2, inp.get("W1s"), inp.get("W3s"), inp.get("W2s"),
                     np.arange(T), I, Is)
    return dict(topk_idx=idx, topk_w=w, Y=Y, **d)
