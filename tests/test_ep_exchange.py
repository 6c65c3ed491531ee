"""Expert-parallel exchange (ep.py) on two gloo ranks on the CPU: the bookkeeping and the
all-to-all row movement around the expert FFN, checked against the oracle's single-GPU
dispatch of all ranks' tokens together.  The row payload is the global token index, so
row ownership and order are visible.  ("Lower latency and higher throughput with
multi-node DeepSeek deployment", Expert Parallelism: Dispatch to the experts' GPUs,
Combine back.)  No GPU: the data plane is torch.distributed, NCCL on GPUs."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle

E, K, T_LOCAL = 16, 3, 37


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _routing(rank):
    rng = np.random.default_rng(100 + rank)
    # a skewed, token-dependent routing: experts 0..3 popular, distinct per token
    p = np.linspace(3, 1, E)
    p /= p.sum()
    return np.stack([rng.choice(E, size=K, replace=False, p=p) for _ in range(T_LOCAL)]).astype(np.int32)


def _worker(rank, world, port, owner_kind, out):
    import torch.distributed as dist

    from expert_routed_ffn_router_gb300 import ep
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        idx = _routing(rank)
        d = oracle.dispatch(idx, E, want_affinity=False)        # this rank's dispatch
        # payload of Xp row r: the global token index of perm[r], and the slot's expert
        gtok = torch.from_numpy(d["perm"].astype(np.float64) + rank * T_LOCAL)
        expert_of_row = np.repeat(np.arange(E), d["counts"])
        Xp = torch.stack([gtok, torch.from_numpy(expert_of_row.astype(np.float64))], 1)
        if owner_kind == "contiguous":
            owner = ep.contiguous_owner(E, world)
        else:
            owner = ep.grouping_owner([(e * 7) % world for e in range(E)], world)   # interleaved
        plan = ep.plan_exchange(torch.from_numpy(d["offsets"]), owner)
        rows = ep.dispatch_rows(Xp, plan)
        # stand-in for the owner's expert FFN: a row-wise function of (token, expert)
        Yp_local = torch.stack([rows[:, 0] * 3.0 + rows[:, 1], rows[:, 1]], 1)
        back = ep.combine_rows(Yp_local, plan, int(d["offsets"][-1]))
        out[rank] = dict(mine=plan.mine.tolist(), recv_counts=plan.recv_counts.numpy(),
                         local_offsets=plan.local_offsets.numpy(), rows=rows.numpy(),
                         Xp=Xp.numpy(), back=back.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("owner_kind", ["contiguous", "grouping"])
def test_exchange_matches_the_single_gpu_dispatch_gloo_world2(owner_kind):
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, owner_kind, out), nprocs=world, join=True)
        res = dict(out)
    # the single-GPU dispatch of every rank's tokens, token t of rank r = r * T_LOCAL + t
    idx_all = np.concatenate([_routing(r) for r in range(world)])
    g = oracle.dispatch(idx_all, E, want_affinity=False)
    seen = []
    for r in range(world):
        R = res[r]
        mine = R["mine"]
        seen += mine
        # counts of my experts from each source rank, and their total = the global count
        for j, e in enumerate(mine):
            per_src = [int((_routing(s) == e).sum()) for s in range(world)]
            assert R["recv_counts"][:, j].tolist() == per_src
            assert R["local_offsets"][j + 1] - R["local_offsets"][j] == g["counts"][e]
            # the owner's rows of expert e are the global permutation's segment of e
            a, b = R["local_offsets"][j], R["local_offsets"][j + 1]
            np.testing.assert_array_equal(R["rows"][a:b, 0], g["perm"][g["offsets"][e]:g["offsets"][e + 1]])
            assert np.all(R["rows"][a:b, 1] == e)
        # every row came back to its source, in Xp order, with the owner's result
        np.testing.assert_array_equal(R["back"][:, 0], R["Xp"][:, 0] * 3.0 + R["Xp"][:, 1])
        np.testing.assert_array_equal(R["back"][:, 1], R["Xp"][:, 1])
    assert sorted(seen) == list(range(E))         # every expert has exactly one owner


def _grace_worker(rank, world, port, group_of, out):
    import torch.distributed as dist

    from expert_routed_ffn_router_gb300 import ep
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        idx = _routing(rank)
        d = oracle.dispatch(idx, E, want_affinity=False)
        gtok = torch.from_numpy(d["perm"].astype(np.float64) + rank * T_LOCAL)
        plan = ep.plan_exchange(torch.from_numpy(d["offsets"]), ep.grouping_owner(group_of, world))
        rows = ep.dispatch_rows(gtok[:, None], plan)
        back = ep.combine_rows(rows * 2.0, plan, int(d["offsets"][-1]))
        out[rank] = dict(mine=plan.mine.tolist(), local_offsets=plan.local_offsets.numpy(),
                         rows=rows[:, 0].numpy(), gtok=gtok.numpy(), back=back[:, 0].numpy())
    finally:
        dist.destroy_process_group()


def test_exchange_over_a_grace_grouping_gloo_world3():
    """Three ranks own the groups of a GRACE-MoE placement computed by the library's planner
    from the co-activation matrix of all ranks' routing (GRACE notes, Core Idea 1: group d
    on GPU d): every rank receives exactly its experts' rows of the single-GPU dispatch,
    and every row comes back to its source."""
    from expert_routed_ffn_router_gb300 import binding as B
    world = 3
    idx_all = np.concatenate([_routing(r) for r in range(world)])
    g = oracle.dispatch(idx_all, E)
    group_of = B.moe_grace_group(g["affinity"], world, 0.5)
    assert sorted(set(group_of.tolist())) == list(range(world))
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_grace_worker, args=(world, port, group_of.tolist(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        R = res[r]
        assert R["mine"] == [e for e in range(E) if group_of[e] == r]
        for j, e in enumerate(R["mine"]):
            a, b = R["local_offsets"][j], R["local_offsets"][j + 1]
            np.testing.assert_array_equal(R["rows"][a:b], g["perm"][g["offsets"][e]:g["offsets"][e + 1]])
        np.testing.assert_array_equal(R["back"], 2.0 * R["gtok"])


def test_owner_helpers():
    from expert_routed_ffn_router_gb300 import ep
    assert ep.contiguous_owner(8, 4).tolist() == [0, 0, 1, 1, 2, 2, 3, 3]
    with pytest.raises(ValueError):
        ep.contiguous_owner(10, 4)
    assert ep.grouping_owner([1, 0, 1], 2).tolist() == [1, 0, 1]
    with pytest.raises(ValueError):
        ep.grouping_owner([0, 2], 2)
