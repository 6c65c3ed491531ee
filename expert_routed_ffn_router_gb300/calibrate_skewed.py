"""Fits the constants of the skewed, correlated routing workload (skewed_recipe.json).

    python -m expert_routed_ffn_router_gb300.calibrate_skewed

The workload: T = 8192 tokens at the DeepSeek-V3 shape; expert e belongs to cluster
e // 32 (8 clusters of 32).  Gate rows and tokens share cluster directions so that a
token's experts come mostly from its own cluster, and a per-expert shift along a common
direction sets each expert's popularity so that the counts follow a Zipf law of exponent
1.2: target count of popularity rank r is min(T, lambda * r^-1.2), with lambda chosen so
that the counts add up to T * K.  Popularity follows the clusters: cluster c holds the
ranks 32c .. 32c + 31 (in the order of the experts' selection biases inside the cluster),
so the popular experts are also the ones that co-activate most.  The shift starts at a
logit of -2 so that the scores sit in the sigmoid's steep range, where every expert can
be reached; a saturated start leaves the low-bias experts unreachable.

This is an input-design tool: it fits `pi` (the per-expert shift) with a fast float64
model of the routing score -- sel = sigmoid(A + pi * D) + bias with A and D precomputed
from the same seeded draws that synth.py makes -- and freezes the constants.  The
library and the oracle never run it; the tests check the resulting workload's counts and
co-activation with the oracle.
"""
from __future__ import annotations

import json
import os

import numpy as np

from . import synth

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "skewed_recipe.json")

N_CLUSTERS = 8
ALPHA = 0.4        # cluster direction in the gate rows (logit boost alpha * gamma = 4)
GAMMA = 10.0       # cluster direction in the tokens
MU = 8.0           # popularity direction in the tokens
ZIPF_S = 1.2


def zipf_targets(T: int, E: int, K: int, s: float = ZIPF_S) -> np.ndarray:
    """Counts by popularity rank: min(T, lam * r^-s) adding up to T*K (bisection on lam)."""
    r = np.arange(1, E + 1, dtype=np.float64)
    lo, hi = 0.0, float(T * K)
    for _ in range(200):
        lam = 0.5 * (lo + hi)
        if np.minimum(T, lam * r ** -s).sum() < T * K:
            lo = lam
        else:
            hi = lam
    return np.minimum(T, hi * r ** -s), hi


def calibrate(iters: int = 400, eta: float = 0.3, verbose: bool = True) -> dict:
    w = synth.workload("skewed")
    T, H, E, K = w.T, w.H, w.E, w.K
    base = synth.workload("skewed", recipe="normal")
    # the noise draws of the routing inputs (identical to synth.routing_inputs)
    r = synth.routing_inputs(base)
    Z = synth.bf16_bits_to_f32(r["X"]).astype(np.float64)
    N = synth.bf16_bits_to_f32(r["W_gate"]).astype(np.float64)
    bias = r["bias"].astype(np.float64)
    # directions (identical to synth._skew)
    rng = synth._rng(w.seed, synth._STREAM["skew"])
    Dm = rng.standard_normal((N_CLUSTERS + 1, H))
    Q, _ = np.linalg.qr(Dm.T)
    U = Q[:, :N_CLUSTERS].T
    d = Q[:, N_CLUSTERS]
    ge = np.arange(E) // (E // N_CLUSTERS)

    targets_by_rank, lam = zipf_targets(T, E, K)
    per = E // N_CLUSTERS
    rank_of = np.empty(E, np.int64)
    for c in range(N_CLUSTERS):
        ex = np.arange(per * c, per * (c + 1))
        rank_of[ex[np.argsort(-bias[ex], kind="stable")]] = np.arange(per * c, per * (c + 1))
    target = targets_by_rank[rank_of]
    mass = np.array([target[ge == c].sum() for c in range(N_CLUSTERS)])

    gt = synth._rng(w.x_seed, synth._STREAM["skew"] + 1).choice(N_CLUSTERS, size=T,
                                                               p=mass / mass.sum())
    X = Z + GAMMA * U[gt] + MU * d[None, :]
    A = X @ (N + ALPHA * U[ge]).T            # T x E, the part of the logit without pi
    D = X @ d                                 # T, coefficient of pi_e

    pi = np.full(E, -2.0 / MU)
    for it in range(iters):
        sel = 1.0 / (1.0 + np.exp(-(A + pi[None, :] * D[:, None]))) + bias[None, :]
        top = np.argpartition(-sel, K, axis=1)[:, :K]
        cnt = np.bincount(top.ravel(), minlength=E).astype(np.float64)
        err = np.log(target + 0.5) - np.log(cnt + 0.5)
        pi += eta * err / MU
        if verbose and (it % 50 == 0 or it == iters - 1):
            print(f"iter {it}: max |log ratio| {np.abs(err).max():.3f}")
    return dict(n_clusters=N_CLUSTERS, alpha=ALPHA, gamma=GAMMA, mu=MU, zipf_s=ZIPF_S,
                zipf_lambda=lam, pi=[float(x) for x in pi],
                cluster_mass=[float(x) for x in mass / mass.sum()],
                popularity="cluster c holds ranks 32c..32c+31, bias order inside a cluster")


def main():
    rec = calibrate()
    with open(OUT, "w") as f:
        json.dump(rec, f, indent=1)
    print("wrote", OUT)


if __name__ == "__main__":
    main()
