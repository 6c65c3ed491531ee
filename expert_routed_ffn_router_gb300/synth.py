"""Seeded synthetic inputs of the layer's workloads.

This module holds the input recipes only -- no step of the method.  The CUDA path and the
oracle both take their inputs from here; the random numbers are drawn here and handed to
both sides.

Recipes (std, not variance, for the normal draws):
  X ~ N(0, 1); W_gate, W1, W3, W2 and the shared expert ~ N(0, 0.02); bias ~ U(-0.1, 0.1)
  (bias = 0 for the prefill workload); values are drawn in fp32 and rounded to bf16 with
  round-to-nearest-even.  Inputs that decide the routing (X, W_gate, bias) are drawn on the
  host with numpy's PCG64, so every machine draws the same routing problem; the expert
  weights of the DeepSeek-V3-sized workloads (22.5 GB) are drawn on the GPU with torch's
  Philox generator, from which the oracle receives copies of the experts it evaluates.

Workloads (DeepSeek-V3 shape: H=7168, E=256, K=8, I=I_shared=2048):
  tiny     T=16, H=256, E=16, K=2, I=I_shared=128, seed 0
  decode   T=128 (64 requests x query length 2), DeepSeek-V3 shape, seed 0
  sweep    T in {2,4,...,256}, DeepSeek-V3 shape; weights seed 0, X seed T
  skewed   T=8192, DeepSeek-V3 shape, 8 clusters of 32 co-activating experts with Zipf
           popularity (gate rows and tokens share cluster directions)
  prefill  T=16384, DeepSeek-V3 shape, bias = 0 (near-uniform routing), seed 0
  profile  T=32, H=7168, E=32, K=8, I=I_shared=2048 (2.8 GB of experts; profiler captures)
  profile_large  T=4096 with the same 32 experts, bias 0 (prefill-like tiles; captures)
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass, replace

import numpy as np

DSV3 = dict(H=7168, E=256, K=8, I=2048, Is=2048)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    K: int
    I: int
    Is: int
    seed: int = 0          # seed of the weights
    x_seed: int = 0        # seed of the token activations
    bias_range: float = 0.1
    recipe: str = "normal"  # "normal" or "skewed"

    def shape(self):
        return dict(T=self.T, H=self.H, E=self.E, K=self.K, I=self.I, I_shared=self.Is)


WORKLOADS = {
    "tiny": Workload("tiny", T=16, H=256, E=16, K=2, I=128, Is=128),
    "decode": Workload("decode", T=128, **DSV3),
    "skewed": Workload("skewed", T=8192, recipe="skewed", **DSV3),
    "prefill": Workload("prefill", T=16384, bias_range=0.0, **DSV3),
}
# small DeepSeek-V3-width case for profiler captures: 32 experts (2.8 GB), same tiles as decode
WORKLOADS["profile"] = Workload("profile", T=32, H=7168, E=32, K=8, I=2048, Is=2048)
# ... and its tensor-bound counterpart: 1024 rows per expert, the tiles of prefill
WORKLOADS["profile_large"] = Workload("profile_large", T=4096, H=7168, E=32, K=8, I=2048,
                                      Is=2048, bias_range=0.0)
SWEEP_T = (2, 4, 8, 16, 32, 64, 128, 256)
for _t in SWEEP_T:
    WORKLOADS[f"sweep{_t}"] = Workload(f"sweep{_t}", T=_t, x_seed=_t, **DSV3)


def workload(name: str, **overrides) -> Workload:
    return replace(WORKLOADS[name], **overrides)


# ----------------------------------------------------------------------------------------
# bf16 encoding of fp32 draws (round to nearest, ties to even)
# ----------------------------------------------------------------------------------------
def f32_to_bf16_bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


_STREAM = dict(X=1, W_gate=2, bias=3, W1=4, W3=5, W2=6, W1s=7, W3s=8, W2s=9,
               skew=10)


# ----------------------------------------------------------------------------------------
# routing inputs (host, numpy)
# ----------------------------------------------------------------------------------------
def _skew_params() -> dict:
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "skewed_recipe.json")
    with open(path) as f:
        return json.load(f)


def routing_inputs(w: Workload) -> dict:
    """X [T,H] and W_gate [E,H] as bf16 bit patterns, bias [E] fp32 (host numpy)."""
    X = _rng(w.x_seed, _STREAM["X"]).standard_normal((w.T, w.H), dtype=np.float32)
    Wg = _rng(w.seed, _STREAM["W_gate"]).standard_normal((w.E, w.H), dtype=np.float32)
    Wg *= np.float32(0.02)
    if w.bias_range > 0:
        bias = _rng(w.seed, _STREAM["bias"]).uniform(-w.bias_range, w.bias_range, w.E)
    else:
        bias = np.zeros(w.E)
    if w.recipe == "skewed":
        X, Wg = _skew(w, X, Wg)
    return dict(X=f32_to_bf16_bits(X), W_gate=f32_to_bf16_bits(Wg),
                bias=bias.astype(np.float32))


def _skew(w: Workload, X: np.ndarray, Wg: np.ndarray):
    """Clustered, popularity-skewed gate rows and tokens.

    Expert e belongs to cluster g(e) = e // (E / n_clusters); u_1..u_n and d are
    orthonormal directions.  Gate rows: W_gate[e] = 0.02 n_e + alpha u_g(e) + pi_e d;
    tokens: X_t = z_t + gamma u_g(t) + mu d, with the cluster of token t drawn from the
    cluster masses.  The constants (alpha, gamma, mu, pi, cluster masses) are frozen in
    skewed_recipe.json."""
    p = _skew_params()
    nc = int(p["n_clusters"])
    r = _rng(w.seed, _STREAM["skew"])
    D = r.standard_normal((nc + 1, w.H))
    Q, _ = np.linalg.qr(D.T)               # H x (nc+1) orthonormal columns
    U = Q[:, :nc].T.astype(np.float32)      # cluster directions
    d = Q[:, nc].astype(np.float32)         # popularity direction
    ge = np.arange(w.E) // (w.E // nc)
    pi = np.asarray(p["pi"], np.float32)
    Wg = Wg + np.float32(p["alpha"]) * U[ge] + pi[:, None] * d[None, :]
    mass = np.asarray(p["cluster_mass"], np.float64)
    gt = _rng(w.x_seed, _STREAM["skew"] + 1).choice(nc, size=w.T, p=mass / mass.sum())
    X = X + np.float32(p["gamma"]) * U[gt] + np.float32(p["mu"]) * d[None, :]
    return X.astype(np.float32), Wg.astype(np.float32)


# ----------------------------------------------------------------------------------------
# expert weights
# ----------------------------------------------------------------------------------------
def expert_weights_host(w: Workload) -> dict:
    """W1, W3 [E,H,I], W2 [E,I,H] and the shared expert as bf16 bit patterns (numpy).
    Use for small workloads only."""
    out = {}
    for name, shp in (("W1", (w.E, w.H, w.I)), ("W3", (w.E, w.H, w.I)),
                      ("W2", (w.E, w.I, w.H)), ("W1s", (w.H, w.Is)), ("W3s", (w.H, w.Is)),
                      ("W2s", (w.Is, w.H))):
        if name.endswith("s") and w.Is == 0:
            out[name] = None
            continue
        a = _rng(w.seed, _STREAM[name]).standard_normal(shp, dtype=np.float32)
        a *= np.float32(0.02)
        out[name] = f32_to_bf16_bits(a)
    return out


def expert_weights_device(w: Workload, device):
    """Tensors of the same shapes and distribution drawn on the GPU with torch's Philox
    generator (bf16 torch tensors); the values differ from expert_weights_host."""
    import torch
    g = torch.Generator(device=device)
    out = {}
    for name, shp in (("W1", (w.E, w.H, w.I)), ("W3", (w.E, w.H, w.I)),
                      ("W2", (w.E, w.I, w.H)), ("W1s", (w.H, w.Is)), ("W3s", (w.H, w.Is)),
                      ("W2s", (w.Is, w.H))):
        if name.endswith("s") and w.Is == 0:
            out[name] = None
            continue
        g.manual_seed(w.seed * 1000 + _STREAM[name])
        t = torch.empty(shp, dtype=torch.bfloat16, device=device)
        if len(shp) == 3:
            for e in range(shp[0]):
                t[e] = (torch.randn(shp[1:], generator=g, device=device,
                                    dtype=torch.float32) * 0.02).to(torch.bfloat16)
        else:
            t.copy_((torch.randn(shp, generator=g, device=device, dtype=torch.float32)
                     * 0.02).to(torch.bfloat16))
        out[name] = t
    return out


def host_inputs(w: Workload) -> dict:
    """Every input of a small workload on the host (numpy)."""
    d = routing_inputs(w)
    d.update(expert_weights_host(w))
    d["K"] = w.K
    return d


def to_device(d: dict, device) -> dict:
    """Upload host numpy inputs as torch tensors (bf16 for uint16 bit patterns)."""
    import torch
    out = {}
    for k, v in d.items():
        if isinstance(v, np.ndarray):
            if v.dtype == np.uint16:
                out[k] = torch.from_numpy(v.view(np.int16).copy()).view(
                    torch.bfloat16).to(device)
            else:
                out[k] = torch.from_numpy(np.ascontiguousarray(v)).to(device)
        else:
            out[k] = v
    return out


def bf16_tensor_to_bits(t) -> np.ndarray:
    """Host uint16 bit patterns of a torch bf16 tensor (copies to the host)."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
