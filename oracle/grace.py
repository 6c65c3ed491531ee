"""Plain numpy oracle of the GRACE-MoE placement steps -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU legs may import this
module; the product path never does.  It shares no code with the C++ planner of the
library (``csrc/grace.cpp``).

Source: the "GRACE-MoE" notes, section "Core Idea":
  1. Expert Grouping -- the affinity matrix A of co-activations, spectral clustering of
     high-affinity experts, controlled non-uniform group sizes [E - delta, E + delta] with
     delta = E * r (E = n / D here called ``ebar``), the intra-group affinity share U(r),
     the group-size deviation S(r), and r chosen at the knee of the curves;
  2. Expert Replication -- the load skew rho = W_max / W_mean, the replica count
     min(max(1, floor(rho)), n_gpu - 1), hot experts of the heaviest group taken by load
     until their cumulative load passes W_max * n_replica / (1 + n_replica), their copies
     on the n_replica least-loaded GPUs;
  3. Routing Policy -- predicted loads W'_max = W_max - W_r + W_p and W'_i = W_i + W_p,
     weights inversely proportional to the predicted load, and the locality order (same
     GPU, then same node, then any node), the weighted choice applying inside a tier.

Readings where the notes leave a step open (also listed in the design notes):
  * spectral clustering is the normalised form: the D leading eigenvectors of
    Deg^-1/2 A Deg^-1/2 (an expert with no co-activation gets degree 1 and keeps a zero
    row), rows scaled to unit length, then a size-bounded k-means on the rows;
  * the integer size bounds are lo = ceil(ebar - delta) and hi = floor(ebar + delta);
  * k-means starts from the farthest-point seeds (first: the expert of largest degree),
    assigns greedily in increasing distance under the upper bound, puts each expert with
    no co-activation into the smallest group (it carries no affinity), then fills groups
    below lo with the cheapest moves from groups above lo; ties go to the lower index;
  * the knee is taken on U(r) over the grid of r (S(r) is reported beside it): with r and
    U scaled to [0, 1], the r where U_scaled - r_scaled is largest -- beyond it a looser
    size bound buys less affinity than on average;
  * an expert's load is its count; the hot experts are the shortest prefix of the heaviest
    group's experts (by load, descending) whose cumulative load exceeds the threshold;
  * W_p = W_r / (1 + n_replica): the hot load spread evenly over the original and the
    copies; the hot experts' instances are the heaviest group's GPU and the replica GPUs.
"""
from __future__ import annotations

import math

import numpy as np


# ------------------------------------------------------------------ Core Idea 1: grouping
def metrics(A: np.ndarray, group_of: np.ndarray, D: int):
    """U = intra-group affinity / all affinity (pairs i < j); S = RMS of |C_d| - n/D."""
    A = np.asarray(A, dtype=np.int64)
    n = A.shape[0]
    total = 0
    intra = 0
    for i in range(n):
        for j in range(i + 1, n):
            total += int(A[i, j])
            if group_of[i] == group_of[j]:
                intra += int(A[i, j])
    U = intra / total if total > 0 else 0.0
    ebar = n / D
    sizes = [int(np.sum(np.asarray(group_of) == d)) for d in range(D)]
    S = math.sqrt(sum((c - ebar) ** 2 for c in sizes) / D)
    return U, S


def size_bounds(n: int, D: int, r: float):
    ebar = n / D
    delta = ebar * r
    lo = max(0, math.ceil(ebar - delta - 1e-12))
    hi = math.floor(ebar + delta + 1e-12)
    return lo, hi


def embedding(A: np.ndarray, D: int) -> np.ndarray:
    """Rows of the D leading eigenvectors of Deg^-1/2 A Deg^-1/2, scaled to unit length."""
    A = np.asarray(A, dtype=np.float64)
    deg = A.sum(1)
    deg[deg <= 0] = 1.0
    s = 1.0 / np.sqrt(deg)
    M = A * s[:, None] * s[None, :]
    w, V = np.linalg.eigh(M)                      # ascending eigenvalues
    Y = V[:, ::-1][:, :D].copy()
    norm = np.linalg.norm(Y, axis=1)
    # an expert with no co-activation has a zero row (up to rounding): it stays at zero
    Y[norm < 1e-9] = 0.0
    norm[norm < 1e-9] = 1.0
    return Y / norm[:, None]


def _assign(Y, C, lo, hi, iso):
    n, D = Y.shape[0], C.shape[0]
    d2 = ((Y[:, None, :] - C[None, :, :]) ** 2).sum(-1)          # [n, D]
    order = sorted(((d2[i, k], i, k) for i in range(n) for k in range(D) if not iso[i]))
    g = np.full(n, -1, np.int64)
    size = np.zeros(D, np.int64)
    for _, i, k in order:
        if g[i] < 0 and size[k] < hi:
            g[i] = k
            size[k] += 1
    # experts with no co-activation: each to the smallest group (lowest id on ties)
    for i in np.nonzero(iso)[0]:
        k = min((kk for kk in range(D) if size[kk] < hi), key=lambda kk: (size[kk], kk))
        g[i] = k
        size[k] += 1
    # groups below lo take the cheapest experts from groups above lo
    while True:
        under = [k for k in range(D) if size[k] < lo]
        if not under:
            break
        k = under[0]
        best = None
        for i in range(n):
            src = g[i]
            if size[src] <= lo:
                continue
            cost = d2[i, k] - d2[i, src]
            if best is None or cost < best[0]:
                best = (cost, i)
        cost, i = best
        size[g[i]] -= 1
        g[i] = k
        size[k] += 1
    return g


def group(A: np.ndarray, D: int, r: float, max_iter: int = 50) -> np.ndarray:
    """Spectral grouping of the experts into D groups of lo..hi experts each."""
    A = np.asarray(A)
    n = A.shape[0]
    lo, hi = size_bounds(n, D, r)
    if lo * D > n or hi * D < n:
        raise ValueError("no partition fits the size bounds")
    Y = embedding(A, D)
    # farthest-point seeds
    deg = np.asarray(A, dtype=np.int64).sum(1)
    seeds = [int(np.argmax(deg))]                  # first maximum: lowest index
    dmin = ((Y - Y[seeds[0]]) ** 2).sum(1)
    while len(seeds) < D:
        cand = dmin.copy()
        cand[seeds] = -1.0
        s = int(np.argmax(cand))
        seeds.append(s)
        dmin = np.minimum(dmin, ((Y - Y[s]) ** 2).sum(1))
    C = Y[seeds].copy()
    iso = deg == 0
    g = _assign(Y, C, lo, hi, iso)
    for _ in range(max_iter):
        C = np.stack([Y[g == k].mean(0) if np.any(g == k) else C[k] for k in range(D)])
        g2 = _assign(Y, C, lo, hi, iso)
        if np.array_equal(g2, g):
            break
        g = g2
    return g.astype(np.int32)


def knee(U, r) -> int:
    """Index of the knee of the utilisation curve U(r) over an increasing grid r: with r
    and U scaled to [0, 1] over the grid, the point where U_scaled - r_scaled is largest
    (beyond it, raising r buys less affinity than it does on average); first maximum."""
    U = np.asarray(U, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)

    def scale(v):
        span = v.max() - v.min()
        return (v - v.min()) / span if span > 0 else np.zeros_like(v)

    d = scale(U) - scale(r)
    return int(np.argmax(d))


def choose_r(A, D: int, r_grid):
    """Groups at every r of the grid, U(r), S(r) and the knee."""
    groups, Us, Ss = [], [], []
    for r in r_grid:
        g = group(A, D, r)
        U, S = metrics(A, g, D)
        groups.append(g)
        Us.append(U)
        Ss.append(S)
    k = knee(Us, r_grid)
    return dict(U=np.array(Us), S=np.array(Ss), knee=k, r=float(r_grid[k]), group_of=groups[k])


# --------------------------------------------------------------- Core Idea 2: replication
def replicate(counts, group_of, D: int):
    """Replica count, hot experts of the heaviest group and the GPUs of their copies."""
    counts = np.asarray(counts, dtype=np.int64)
    group_of = np.asarray(group_of)
    W = [int(counts[group_of == d].sum()) for d in range(D)]
    W_mean = sum(W) / D
    heavy = max(range(D), key=lambda d: (W[d], -d))          # ties: lower group
    W_max = W[heavy]
    rho = W_max / W_mean if W_mean > 0 else 0.0
    n_rep = min(max(1, math.floor(rho)), D - 1)
    members = [e for e in range(len(counts)) if group_of[e] == heavy]
    members.sort(key=lambda e: (-counts[e], e))
    thr = W_max * n_rep / (1 + n_rep)
    hot, acc = [], 0
    for e in members:                             # until the cumulative load exceeds thr
        if acc > thr:
            break
        hot.append(e)
        acc += int(counts[e])
    others = sorted((d for d in range(D) if d != heavy), key=lambda d: (W[d], d))
    replicas = others[:n_rep]
    return dict(W=W, W_mean=W_mean, W_max=W_max, heaviest=heavy, rho=rho, n_replica=n_rep,
                hot=hot, W_r=acc, replica_gpus=replicas)


# ----------------------------------------------------------------- Core Idea 3: routing
def route_table(rep: dict, gpus_per_node: int):
    """Instance weights of a hot expert for a token on each source GPU.

    Instances: [heaviest group's GPU] + replica GPUs.  Predicted loads W'_max = W_max -
    W_r + W_p for the original, W'_i = W_i + W_p for a replica GPU, W_p = W_r / (1 +
    n_replica); weight proportional to 1 / W'.  A token takes the instance on its own GPU
    if there is one, else the instances on its node, else all instances."""
    inst = [rep["heaviest"]] + list(rep["replica_gpus"])
    W_p = rep["W_r"] / (1 + rep["n_replica"])
    pred = [rep["W_max"] - rep["W_r"] + W_p] + [rep["W"][g] + W_p for g in rep["replica_gpus"]]
    inv = [1.0 / p if p > 0 else 1.0 for p in pred]
    D = len(rep["W"])
    table = np.zeros((D, len(inst)))
    for src in range(D):
        tier = [k for k, g in enumerate(inst) if g == src]
        if not tier:
            tier = [k for k, g in enumerate(inst) if g // gpus_per_node == src // gpus_per_node]
        if not tier:
            tier = list(range(len(inst)))
        z = sum(inv[k] for k in tier)
        for k in tier:
            table[src, k] = inv[k] / z
    return dict(instances=inst, predicted=pred, table=table)
