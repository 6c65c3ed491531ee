"""Shared helpers of the GPU parity tests: build seeded inputs on the device, run the CUDA
path through the C ABI, and compute the oracle's answer on the host."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from expert_routed_ffn_router_gb300 import binding as B
from expert_routed_ffn_router_gb300 import synth

DEV = "cuda:0"
# Tolerances of the floating-point outputs (the integer outputs must be bit-exact):
Y_REL_FROB = 5e-3      # relative Frobenius error of Y
Y_MAX_ABS = 3e-2       # max abs error of Y
W_MAX_ABS = 1e-5       # routing weights


def rel_frob(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_tensor_to_bits(t)


def host_to_device_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(DEV)


class Problem:
    """One layer problem: host copies of the routing inputs, device copies of everything."""

    def __init__(self, w: synth.Workload, routing: dict | None = None, weights_dev=None,
                 host_weights: bool | None = None, opts: dict | None = None):
        self.w = w
        self.opts = opts          # routing options (keywords of oracle.router_ex), or None
        self.routing = routing if routing is not None else synth.routing_inputs(w)
        small = w.E * w.H * w.I < 64 * 1024 * 1024
        if host_weights is None:
            host_weights = small
        if weights_dev is not None:
            self.dev = dict(weights_dev)
            self.host_w = None
        elif host_weights:
            self.host_w = synth.expert_weights_host(w)
            self.dev = {k: (None if v is None else host_to_device_bf16(v))
                        for k, v in self.host_w.items()}
        else:
            self.host_w = None
            self.dev = synth.expert_weights_device(w, DEV)
        self.dev["W_gate"] = host_to_device_bf16(self.routing["W_gate"])
        self.dev["bias"] = torch.from_numpy(self.routing["bias"]).to(DEV)
        self.X = host_to_device_bf16(self.routing["X"])

    def expert_host(self, name: str, e: int | None = None) -> np.ndarray:
        if self.host_w is not None:
            a = self.host_w[name]
            return a if e is None else a[e]
        t = self.dev[name]
        return bits(t if e is None else t[e])

    # ---------------------------------------------------------------- CUDA path
    def run_layer(self, with_affinity=True):
        layer = B.MoELayer(self.dev, self.w.T, self.w.K, with_affinity=with_affinity,
                           routing=self.opts)
        layer.forward(self.X)
        torch.cuda.synchronize()
        st = layer.status()
        assert st == 0, f"device status {st}"
        return layer

    # ------------------------------------------------------------------- oracle
    def oracle_routing(self):
        if self.opts:
            return oracle.router_ex(self.routing["X"], self.routing["W_gate"],
                                    self.routing["bias"], self.w.K, **self.opts)
        return oracle.router(self.routing["X"], self.routing["W_gate"], self.routing["bias"],
                             self.w.K)

    def oracle_Y(self, idx, wts, tokens) -> np.ndarray:
        """Y of the listed tokens, evaluated by the oracle expert by expert (only a few
        experts' weights are copied to the host at a time)."""
        sh = None
        if self.w.Is > 0:
            sh = tuple(self.expert_host(n) for n in ("W1s", "W3s", "W2s"))
        fetch = lambda e: tuple(self.expert_host(n, e) for n in ("W1", "W3", "W2"))
        return oracle.layer_tokens_by_expert(self.routing["X"], idx, wts, fetch, sh, tokens,
                                             self.w.I, self.w.Is)


def covering_tokens(idx: np.ndarray, n: int) -> list:
    """At least n tokens (all of them when T <= n) such that every expert some token chose
    appears: for each chosen expert, in increasing order, the first token choosing it;
    then evenly spaced tokens up to n, plus the first and the last token."""
    T = idx.shape[0]
    if T <= n:
        return list(range(T))
    first = {}
    for t in range(T):
        for e in idx[t]:
            first.setdefault(int(e), t)
    chosen = set(first.values()) | {0, T - 1}
    for t in np.linspace(0, T - 1, n).astype(int):
        if len(chosen) >= n:
            break
        chosen.add(int(t))
    return sorted(chosen)


def check_dispatch(layer, X: torch.Tensor, d: dict):
    """The layer's own dispatch results (offsets, perm, slot_pos and Xp in its workspace)
    against the oracle's dispatch of the same routing: bit-exact."""
    inter = layer.intermediates()
    assert np.array_equal(inter["offsets"].cpu().numpy(), d["offsets"]), "offsets differ"
    perm_g = inter["perm"].cpu().numpy()
    bad = np.nonzero(perm_g != d["perm"])[0]
    assert bad.size == 0, f"perm differs at rows {bad[:10]}"
    slot_g = inter["slot_pos"].cpu().numpy()
    assert np.array_equal(slot_g, d["slot_pos"]), "slot_pos differs"
    perm_o = torch.from_numpy(d["perm"].astype(np.int64)).to(X.device)
    assert torch.equal(inter["Xp"].view(torch.int16), X.view(torch.int16)[perm_o]), "Xp != X[perm]"


def check_layer(p: Problem, tokens=None, check_affinity=True, n_cover=None):
    """Full-layer parity: routing, counts, the dispatch bookkeeping (offsets, perm,
    slot_pos, Xp) and affinity bit-exact over all tokens; Y on `tokens` (all tokens when
    None, or with n_cover set, covering_tokens(n_cover)) within the stated tolerances."""
    layer = p.run_layer(with_affinity=check_affinity)
    idx_o, w_o = p.oracle_routing()
    idx_g = layer.topk_idx.cpu().numpy()
    bad = np.nonzero((idx_g != idx_o).any(1))[0]
    assert bad.size == 0, f"top-k differs on tokens {bad[:10]}: gpu {idx_g[bad[:3]]} oracle {idx_o[bad[:3]]}"
    w_err = np.abs(layer.topk_w.cpu().numpy().astype(np.float64) - w_o).max()
    assert w_err <= W_MAX_ABS, w_err
    d = oracle.dispatch(idx_o, p.w.E, want_affinity=check_affinity)
    assert np.array_equal(layer.counts.cpu().numpy(), d["counts"])
    check_dispatch(layer, p.X, d)
    if check_affinity:
        assert np.array_equal(layer.affinity.cpu().numpy(), d["affinity"])
    if n_cover is not None:
        tokens = covering_tokens(idx_o, n_cover)
    elif tokens is None:
        tokens = np.arange(p.w.T)
    tokens = np.asarray(tokens)
    Y_o = p.oracle_Y(idx_o, w_o, tokens)
    Y_g = layer.Y.cpu().numpy()[tokens].astype(np.float64)
    rf = rel_frob(Y_g, Y_o)
    ma = float(np.abs(Y_g - Y_o).max())
    assert rf <= Y_REL_FROB and ma <= Y_MAX_ABS, (rf, ma)
    return dict(layer=layer, rel_frob=rf, max_abs=ma, idx=idx_o, w=w_o, disp=d, tokens=tokens)
