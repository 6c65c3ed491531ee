"""Pins of the GRACE-MoE placement oracle (``oracle/grace.py``) against worked numbers,
closed forms and invariants ("GRACE-MoE" notes, Core Idea 1-3).  CPU only."""

import numpy as np
import pytest

from oracle import grace


def _sym(n, pairs):
    A = np.zeros((n, n), np.int32)
    for (i, j), v in pairs.items():
        A[i, j] = A[j, i] = v
    return A


def _planted(blocks, size, seed, intra=(40, 80), cross=(0, 3)):
    """Block-structured co-activation counts: strong inside a block, weak across."""
    rng = np.random.default_rng(seed)
    n = blocks * size
    A = rng.integers(cross[0], cross[1] + 1, (n, n))
    for b in range(blocks):
        s = slice(b * size, (b + 1) * size)
        A[s, s] = rng.integers(intra[0], intra[1] + 1, (size, size))
    A = np.triu(A, 1)
    return (A + A.T).astype(np.int32)


def _same_partition(g1, g2):
    pairs = {}
    for a, b in zip(g1, g2):
        if pairs.setdefault(int(a), int(b)) != int(b):
            return False
    return len(set(pairs.values())) == len(pairs)


# ------------------------------------------------------------------ U(r), S(r)
def test_metrics_worked_example():
    # pairs (0,1)=5, (2,3)=3, (0,2)=1, (1,3)=1: total 10
    A = _sym(4, {(0, 1): 5, (2, 3): 3, (0, 2): 1, (1, 3): 1})
    U, S = grace.metrics(A, np.array([0, 0, 1, 1]), 2)
    assert U == pytest.approx(0.8, abs=1e-15) and S == 0.0
    U, S = grace.metrics(A, np.array([0, 0, 0, 1]), 2)      # (0,1)+(0,2) = 6 of 10
    assert U == pytest.approx(0.6, abs=1e-15) and S == pytest.approx(1.0, abs=1e-15)
    U, S = grace.metrics(A, np.array([0, 1, 2, 3]), 4)      # singletons: nothing intra
    assert U == 0.0 and S == 0.0


def test_size_bounds_worked_example():
    assert grace.size_bounds(256, 8, 0.0) == (32, 32)
    assert grace.size_bounds(256, 8, 0.25) == (24, 40)     # 32 -+ 8
    assert grace.size_bounds(10, 4, 0.1) == (3, 2)          # 2.5 -+ 0.25: no integer fits
    assert grace.size_bounds(10, 4, 0.2) == (2, 3)


# ------------------------------------------------------------------ spectral embedding
def test_embedding_of_disconnected_blocks_is_one_point_per_block():
    # D disconnected blocks: the leading eigenvalue 1 has multiplicity D and its eigenspace
    # is spanned by the blocks' sqrt-degree vectors, so after row scaling every expert of
    # a block maps to the same unit vector and different blocks to orthogonal ones
    A = _planted(4, 6, seed=1, cross=(0, 0))
    Y = grace.embedding(A, 4)
    G = Y @ Y.T
    blk = np.arange(24) // 6
    same = blk[:, None] == blk[None, :]
    np.testing.assert_allclose(G[same], 1.0, atol=1e-9)
    np.testing.assert_allclose(G[~same], 0.0, atol=1e-9)


# -------------------------------------------------------------------------- grouping
@pytest.mark.parametrize("blocks,size", [(8, 32), (4, 8), (2, 16)])
def test_planted_groups_are_recovered(blocks, size):
    A = _planted(blocks, size, seed=blocks + size)
    g = grace.group(A, blocks, 0.0)
    assert _same_partition(g, np.arange(blocks * size) // size)
    U, S = grace.metrics(A, g, blocks)
    U_planted, _ = grace.metrics(A, np.arange(blocks * size) // size, blocks)
    assert U == U_planted and S == 0.0


@pytest.mark.parametrize("r", [0.0, 0.1, 0.25, 0.5])
def test_group_sizes_respect_the_bounds(r):
    rng = np.random.default_rng(3)
    A = rng.integers(0, 20, (48, 48))
    A = np.triu(A, 1)
    A = (A + A.T).astype(np.int32)
    g = grace.group(A, 6, r)
    lo, hi = grace.size_bounds(48, 6, r)
    sizes = np.bincount(g, minlength=6)
    assert sizes.sum() == 48 and sizes.min() >= lo and sizes.max() <= hi


def test_unequal_planted_groups_need_a_nonzero_r():
    # blocks of 12, 12, 4, 4 experts (mean 8): r = 0 forces 8 per group and splits the
    # big blocks; r = 0.5 (sizes 4..12) keeps every block whole
    sizes = [12, 12, 4, 4]
    blk = np.repeat(np.arange(4), sizes)
    rng = np.random.default_rng(4)
    A = np.where(blk[:, None] == blk[None, :], rng.integers(40, 80, (32, 32)),
                 rng.integers(0, 2, (32, 32)))
    A = np.triu(A, 1)
    A = (A + A.T).astype(np.int32)
    g0 = grace.group(A, 4, 0.0)
    g5 = grace.group(A, 4, 0.5)
    assert np.all(np.bincount(g0, minlength=4) == 8)
    assert _same_partition(g5, blk)
    assert grace.metrics(A, g5, 4)[0] > grace.metrics(A, g0, 4)[0]


def test_grouping_follows_a_relabelling_of_the_experts():
    A = _planted(4, 8, seed=5)
    p = np.random.default_rng(6).permutation(32)
    g = grace.group(A, 4, 0.0)
    gp = grace.group(A[np.ix_(p, p)], 4, 0.0)
    assert _same_partition(gp, g[p])


# ------------------------------------------------------------------------------ knee
def test_knee_of_a_curve_with_one_corner():
    r = [0.0, 0.1, 0.2, 0.3, 0.4]
    assert grace.knee([0.0, 0.9, 0.95, 0.97, 1.0], r) == 1           # saturates after 0.1
    assert grace.knee([0.5, 0.8, 0.9, 0.93, 0.95], r) == 1
    assert grace.knee([0.0, 0.1, 0.2, 0.9, 1.0], r) == 3             # late jump
    assert grace.knee([0.5, 0.5, 0.5], [0.0, 1.0, 2.0]) == 0         # flat: first point


def test_choose_r_on_unequal_blocks_picks_a_grid_point_that_keeps_the_blocks():
    sizes = [12, 12, 4, 4]
    blk = np.repeat(np.arange(4), sizes)
    rng = np.random.default_rng(7)
    A = np.where(blk[:, None] == blk[None, :], rng.integers(40, 80, (32, 32)),
                 rng.integers(0, 2, (32, 32)))
    A = np.triu(A, 1)
    A = (A + A.T).astype(np.int32)
    res = grace.choose_r(A, 4, [0.0, 0.125, 0.25, 0.375, 0.5, 0.75])
    assert np.all(np.diff(res["U"]) >= -1e-12)        # looser size bounds never lose affinity
    assert res["r"] == 0.5 and _same_partition(res["group_of"], blk)


# ----------------------------------------------------------------------- replication
def _counts_for(groups_loads):
    counts, group_of = [], []
    for d, loads in enumerate(groups_loads):
        counts += loads
        group_of += [d] * len(loads)
    return np.array(counts), np.array(group_of)


def test_replication_worked_example():
    # W = [100, 40, 30, 30]: mean 50, rho = 2, n_replica = min(max(1, 2), 3) = 2;
    # threshold 100 * 2 / 3 = 66.7: loads 50 then 70 > 66.7 -> two hot experts, W_r = 70;
    # copies on the two least-loaded other GPUs, 2 and 3 (equal loads: lower first)
    counts, group_of = _counts_for([[20, 50, 10, 20], [40], [30], [30]])
    rep = grace.replicate(counts, group_of, 4)
    assert rep["W"] == [100, 40, 30, 30] and rep["heaviest"] == 0
    assert rep["rho"] == 2.0 and rep["n_replica"] == 2
    assert rep["hot"] == [1, 0] and rep["W_r"] == 70      # equal loads 20, 20: lower index
    assert rep["replica_gpus"] == [2, 3]


def test_replication_count_is_capped():
    # one group holds everything: rho = D, capped at n_gpu - 1
    counts, group_of = _counts_for([[100, 100], [0], [0], [0]])
    rep = grace.replicate(counts, group_of, 4)
    assert rep["rho"] == 4.0 and rep["n_replica"] == 3
    # perfectly balanced: rho = 1 -> one replica
    counts, group_of = _counts_for([[10], [10], [10], [10]])
    assert grace.replicate(counts, group_of, 4)["n_replica"] == 1


# --------------------------------------------------------------------------- routing
def test_route_table_worked_example():
    # W = [100, 10, 40, 50]: rho = 2, 2 replicas on GPUs 1 and 2; hot loads 60 then 90 >
    # 66.7 -> W_r = 90, W_p = 30; predicted [100 - 90 + 30, 10 + 30, 40 + 30] = [40, 40, 70]
    counts, group_of = _counts_for([[60, 30, 10], [10], [40], [50]])
    rep = grace.replicate(counts, group_of, 4)
    assert rep["replica_gpus"] == [1, 2] and rep["W_r"] == 90
    one_node = grace.route_table(rep, gpus_per_node=4)
    assert one_node["instances"] == [0, 1, 2]
    np.testing.assert_allclose(one_node["predicted"], [40.0, 40.0, 70.0])
    np.testing.assert_allclose(one_node["table"][3], [7 / 18, 7 / 18, 4 / 18], rtol=1e-14)
    np.testing.assert_allclose(one_node["table"][0], [1, 0, 0])        # own GPU first
    np.testing.assert_allclose(one_node["table"][2], [0, 0, 1])
    two_nodes = grace.route_table(rep, gpus_per_node=2)
    np.testing.assert_allclose(two_nodes["table"][3], [0, 0, 1])       # node 1 holds GPU 2
    np.testing.assert_allclose(two_nodes["table"][1], [0, 1, 0])
    eight = grace.route_table(rep, gpus_per_node=1)
    np.testing.assert_allclose(eight["table"][3], [7 / 18, 7 / 18, 4 / 18], rtol=1e-14)


def test_route_table_rows_are_distributions():
    rng = np.random.default_rng(8)
    counts = rng.integers(0, 500, 64)
    group_of = np.repeat(np.arange(8), 8)
    rep = grace.replicate(counts, group_of, 8)
    t = grace.route_table(rep, gpus_per_node=4)["table"]
    np.testing.assert_allclose(t.sum(1), 1.0, atol=1e-14)
    assert np.all(t >= 0)


# ------------------------------------------------- experts with no co-activation at all
def _blocks_and_isolated(block_sizes, n_isolated, v=10):
    n = sum(block_sizes) + n_isolated
    A = np.zeros((n, n), np.int32)
    start = 0
    for b in block_sizes:
        A[start:start + b, start:start + b] = v
        start += b
    np.fill_diagonal(A, 0)
    return A


@pytest.mark.parametrize("block_sizes,r,expected", [
    # blocks {0,1,2} and {3,4,5}; isolated 6 and 7.  Both groups hold 3 experts when the
    # isolated ones are placed: 6 goes to the lower group id, then 7 to the other group
    ((3, 3), 0.5, [0, 0, 0, 1, 1, 1, 0, 1]),
    # blocks {0,1,2,3} and {4,5}: the smaller group takes both isolated experts
    ((4, 2), 0.5, [0, 0, 0, 0, 1, 1, 1, 1]),
    ((4, 2), 0.0, [0, 0, 0, 0, 1, 1, 1, 1]),
])
def test_isolated_experts_join_the_smallest_group(block_sizes, r, expected):
    # An expert that no token co-activates with another has a zero row in A: its spectral
    # embedding row is zero (rounding noise only), so its position carries no affinity.
    # The grouping's reading places each such expert, in index order, into the group that
    # is smallest at that moment (lower group id on ties).  Worked by hand: the D = 2
    # leading eigenvectors span the two blocks' indicator vectors, every block maps to one
    # unit vector and the blocks become the groups (first seed: the expert of largest
    # degree, i.e. expert 0; second: the farthest point, a member of the other block).
    A = _blocks_and_isolated(block_sizes, 2)
    g = grace.group(A, 2, r)
    assert _same_partition(g, np.array(expected)), g.tolist()
    assert g[6] != g[7] if block_sizes == (3, 3) else g[6] == g[7] == g[4]
    U, _ = grace.metrics(A, g, 2)
    assert U == 1.0                      # every co-activation stays inside a group
