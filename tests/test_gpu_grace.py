"""GRACE-MoE placement planned from the by-products the GPU layer emits (counts and the
co-activation matrix of the skewed, clustered workload), against the placement oracle fed
the oracle's own by-products ("GRACE-MoE" notes, Core Idea 1-3)."""
import numpy as np
import pytest

import oracle
from oracle import grace
from expert_routed_ffn_router_gb300 import binding as B
from expert_routed_ffn_router_gb300 import synth

from gpu_common import Problem

pytestmark = pytest.mark.gpu


def _same_partition(g1, g2):
    m = {}
    for a, b in zip(g1, g2):
        if m.setdefault(int(a), int(b)) != int(b):
            return False
    return len(set(m.values())) == len(m)


def test_plan_from_the_layer_by_products():
    w = synth.workload("skewed", T=1024)
    p = Problem(w, host_weights=False)
    layer = p.run_layer(with_affinity=True)
    A_gpu = layer.affinity.cpu().numpy()
    c_gpu = layer.counts.cpu().numpy()
    idx, _ = p.oracle_routing()
    d = oracle.dispatch(idx, w.E)
    assert np.array_equal(A_gpu, d["affinity"]) and np.array_equal(c_gpu, d["counts"])
    grid = [0.0, 0.125, 0.25, 0.5]
    lib = B.moe_grace_choose_r(A_gpu, 8, grid)
    ref = grace.choose_r(d["affinity"], 8, grid)
    assert lib["knee"] == ref["knee"] and _same_partition(lib["group_of"], ref["group_of"])
    rep = B.moe_grace_replicate(c_gpu, lib["group_of"], 8)
    rref = grace.replicate(d["counts"], lib["group_of"], 8)
    for k in ("W", "heaviest", "n_replica", "hot", "W_r", "replica_gpus"):
        assert rep[k] == rref[k], k
    t = B.moe_grace_route_table(rep, 4)["table"]
    np.testing.assert_allclose(t, grace.route_table(rref, 4)["table"], rtol=1e-14, atol=0)
