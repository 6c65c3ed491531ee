"""The library's GRACE-MoE planner (C ABI, host code) against the placement oracle
("GRACE-MoE" notes, Core Idea 1-3) on the same inputs.  CPU only: the planner runs on the
host.  Integer-defined results must match exactly; groupings are compared as partitions
(group ids are labels)."""
import numpy as np
import pytest

import oracle
from oracle import grace
from expert_routed_ffn_router_gb300 import binding as B
from expert_routed_ffn_router_gb300 import synth


def _random_affinity(n, seed, hi=30):
    rng = np.random.default_rng(seed)
    A = np.triu(rng.integers(0, hi, (n, n)), 1)
    return (A + A.T).astype(np.int32)


def _planted(sizes, seed):
    blk = np.repeat(np.arange(len(sizes)), sizes)
    n = len(blk)
    rng = np.random.default_rng(seed)
    A = np.where(blk[:, None] == blk[None, :], rng.integers(40, 80, (n, n)),
                 rng.integers(0, 3, (n, n)))
    A = np.triu(A, 1)
    return (A + A.T).astype(np.int32), blk


def _same_partition(g1, g2):
    m = {}
    for a, b in zip(g1, g2):
        if m.setdefault(int(a), int(b)) != int(b):
            return False
    return len(set(m.values())) == len(m)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_metrics_match(seed):
    A = _random_affinity(40, seed)
    g = np.random.default_rng(seed + 10).integers(0, 5, 40).astype(np.int32)
    assert B.moe_grace_metrics(A, g, 5) == grace.metrics(A, g, 5)


@pytest.mark.parametrize("sizes,r", [([32] * 8, 0.0), ([12, 12, 4, 4], 0.5), ([8] * 4, 0.25),
                                     ([20, 10, 10, 8], 0.7)])
def test_grouping_matches_on_planted_blocks(sizes, r):
    A, blk = _planted(sizes, seed=len(sizes) + sum(sizes))
    g_lib = B.moe_grace_group(A, len(sizes), r)
    g_ref = grace.group(A, len(sizes), r)
    assert _same_partition(g_lib, g_ref)
    assert _same_partition(g_lib, blk)


@pytest.mark.parametrize("n,D,r", [(48, 6, 0.0), (48, 6, 0.25), (64, 8, 0.5), (30, 4, 0.2)])
def test_grouping_matches_on_random_affinity(n, D, r):
    A = _random_affinity(n, seed=n + D)
    g_lib = B.moe_grace_group(A, D, r)
    g_ref = grace.group(A, D, r)
    lo, hi = grace.size_bounds(n, D, r)
    sizes = np.bincount(g_lib, minlength=D)
    assert sizes.min() >= lo and sizes.max() <= hi
    assert _same_partition(g_lib, g_ref)


def test_choose_r_matches():
    A, blk = _planted([12, 12, 4, 4], seed=9)
    grid = [0.0, 0.125, 0.25, 0.375, 0.5, 0.75]
    lib = B.moe_grace_choose_r(A, 4, grid)
    ref = grace.choose_r(A, 4, grid)
    assert lib["knee"] == ref["knee"] and lib["r"] == 0.5
    np.testing.assert_allclose(lib["U"], ref["U"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lib["S"], ref["S"], rtol=0, atol=1e-15)
    assert _same_partition(lib["group_of"], blk)


@pytest.mark.parametrize("seed,D", [(0, 8), (1, 4), (2, 16), (3, 2)])
def test_replication_and_route_table_match(seed, D):
    rng = np.random.default_rng(seed)
    E = 64
    counts = (rng.zipf(1.5, E) * 10).clip(0, 100000).astype(np.int32)
    group_of = rng.permutation(np.arange(E) % D).astype(np.int32)
    lib = B.moe_grace_replicate(counts, group_of, D)
    ref = grace.replicate(counts, group_of, D)
    for k in ("W", "heaviest", "n_replica", "hot", "W_r", "replica_gpus", "W_max"):
        assert lib[k] == ref[k], k
    assert lib["rho"] == ref["rho"] and lib["W_mean"] == ref["W_mean"]
    for gpn in (1, 2, 4, D):
        tl = B.moe_grace_route_table(lib, gpn)
        tr = grace.route_table(ref, gpn)
        assert tl["instances"] == tr["instances"]
        np.testing.assert_allclose(tl["predicted"], tr["predicted"], rtol=1e-15)
        np.testing.assert_allclose(tl["table"], tr["table"], rtol=1e-14, atol=0)


def test_skewed_routing_groups_follow_the_clusters():
    # co-activations of 1024 tokens of the skewed workload (8 clusters of 32 experts),
    # routed by the oracle: the planner and the oracle agree, and the grouping at the knee
    # keeps as much co-activation inside groups as the clusters the inputs were built from
    # (r = 0, every group exactly 32, keeps less: the two experts almost every token picks
    # hold ~45% of all co-activations and sit between the clusters)
    w = synth.workload("skewed", T=1024)
    r = synth.routing_inputs(w)
    idx, _ = oracle.router(r["X"], r["W_gate"], r["bias"], w.K)
    d = oracle.dispatch(idx, w.E)
    A, counts = d["affinity"], d["counts"]
    grid = [0.0, 0.125, 0.25, 0.5]
    lib = B.moe_grace_choose_r(A, 8, grid)
    ref = grace.choose_r(A, 8, grid)
    assert lib["knee"] == ref["knee"]
    np.testing.assert_allclose(lib["U"], ref["U"], rtol=0, atol=1e-12)
    assert _same_partition(lib["group_of"], ref["group_of"])
    U_clusters, _ = grace.metrics(A, np.arange(w.E) // 32, 8)
    assert lib["knee"] > 0 and lib["U"][lib["knee"]] >= U_clusters - 0.02
    rep = B.moe_grace_replicate(counts, lib["group_of"], 8)
    assert rep["hot"] == grace.replicate(counts, lib["group_of"], 8)["hot"]


@pytest.mark.parametrize("block_sizes,r", [((3, 3), 0.5), ((4, 2), 0.5), ((4, 2), 0.0)])
def test_isolated_experts_are_placed_like_the_oracle(block_sizes, r):
    # experts with no co-activation (zero rows of A) go to the smallest group, as the
    # oracle's reading places them (pinned by hand in test_grace_oracle)
    n = sum(block_sizes) + 2
    A = np.zeros((n, n), np.int32)
    s = 0
    for b in block_sizes:
        A[s:s + b, s:s + b] = 10
        s += b
    np.fill_diagonal(A, 0)
    g_lib = B.moe_grace_group(A, 2, r)
    g_ref = grace.group(A, 2, r)
    assert _same_partition(g_lib, g_ref), (g_lib.tolist(), g_ref.tolist())
