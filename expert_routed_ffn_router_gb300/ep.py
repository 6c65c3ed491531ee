"""Expert parallelism: the row exchange around the expert FFN when the experts of a layer
are spread over several GPUs.

"Lower latency and higher throughput with multi-node DeepSeek deployment", section
"Expert Parallelism": each GPU holds a subset of the routed experts; Dispatch sends every
token to the GPUs of its experts before the expert GEMMs and Combine brings the results
back for the weighted sum.  On one GPU these are the library's moe_dispatch and moe_combine;
across GPUs the exchange below sits between them:

  1. every rank runs the router and moe_dispatch on its own tokens: Xp rows ordered by
     (expert, local token), with per-expert counts;
  2. counts exchange: each rank sends every other rank the counts of the experts that rank
     owns (one all-to-all of a few integers);
  3. rows exchange (the Dispatch): all-to-all with splits, each rank sending the rows of
     the experts another rank owns, in expert order;
  4. the owner regroups the rows it received by (local expert, source rank) and runs the
     grouped FFN (moe_expert_ffn) over its experts;
  5. rows back (the Combine's exchange): the transposed all-to-all, after which every rank
     holds the FFN output of each of its Xp rows in Xp order;
  6. moe_combine on every rank, as on one GPU.

Within an expert, rows end up ordered by source rank and then by the source's token order:
with global token index = rank * tokens_per_rank + local index, that is the single-GPU
dispatch's order (ascending token), so the owner's rows of an expert are exactly the
single-GPU permutation's segment of that expert.

The data plane is torch.distributed (NCCL on GPUs, gloo for the CPU tests); the row
gathers are index selects of whole rows.  Expert ownership: contiguous ranges of E/W
experts (the pages' EP partitioning), or the groups of a GRACE-MoE placement (Core Idea 1:
group d on rank d).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.distributed as dist


def contiguous_owner(E: int, world: int) -> torch.Tensor:
    """owner[e] for consecutive ranges of E / world experts per rank."""
    if world < 1 or E % world:
        raise ValueError("E must be a multiple of the number of ranks")
    return torch.arange(E, dtype=torch.int64) // (E // world)


def grouping_owner(group_of, world: int) -> torch.Tensor:
    """owner[e] = group_of[e]: a placement's groups, group d on rank d."""
    g = torch.as_tensor(group_of, dtype=torch.int64)
    if g.numel() and (int(g.min()) < 0 or int(g.max()) >= world):
        raise ValueError("group ids must lie in [0, world)")
    return g


@dataclass
class ExchangePlan:
    """Bookkeeping of one exchange (as seen by one rank)."""
    owner: torch.Tensor          # [E] rank of each expert
    mine: torch.Tensor           # my experts, ascending
    send_order: torch.Tensor     # Xp row indices in send order (by destination, then expert)
    send_splits: list            # rows sent to each rank
    recv_counts: torch.Tensor    # [world, len(mine)] rows of each of my experts from each rank
    recv_splits: list            # rows received from each rank
    local_order: torch.Tensor    # received row indices regrouped by (my expert, source rank)
    local_offsets: torch.Tensor  # [len(mine) + 1] row offsets of my experts after regrouping


def _world(group):
    return dist.get_world_size(group), dist.get_rank(group)


def plan_exchange(offsets: torch.Tensor, owner: torch.Tensor, group=None) -> ExchangePlan:
    """Steps 2 and the bookkeeping of 3-5 from this rank's dispatch offsets [E + 1] (rows of
    expert e are offsets[e] .. offsets[e+1] of Xp).  Collective: every rank calls it."""
    world, rank = _world(group)
    # the counts travel on the offsets' device (NCCL exchanges device tensors only, gloo
    # host ones); the bookkeeping below is host work on a few integers per expert
    dev = offsets.device
    offsets = offsets.to(torch.int64).cpu()
    owner = owner.to(torch.int64).cpu()
    counts = offsets[1:] - offsets[:-1]
    experts_of = [torch.nonzero(owner == d).flatten() for d in range(world)]
    mine = experts_of[rank]
    # 2. counts exchange: to rank d, the counts of d's experts (ascending)
    send_c = torch.cat([counts[experts_of[d]] for d in range(world)]).to(dev)
    recv_c = torch.empty(world * mine.numel(), dtype=torch.int64, device=dev)
    dist.all_to_all_single(recv_c, send_c, [mine.numel()] * world,
                           [experts_of[d].numel() for d in range(world)], group=group)
    recv_counts = recv_c.cpu().view(world, mine.numel())
    # 3. send order: by destination, then by expert (the expert's Xp rows in order)
    order = []
    send_splits = []
    for d in range(world):
        n = 0
        for e in experts_of[d].tolist():
            a, b = int(offsets[e]), int(offsets[e + 1])
            order.append(torch.arange(a, b, dtype=torch.int64))
            n += b - a
        send_splits.append(n)
    send_order = torch.cat(order) if order else torch.zeros(0, dtype=torch.int64)
    recv_splits = recv_counts.sum(1).tolist()
    # 4. received rows come as [source rank][my expert] blocks: regroup expert-major
    src_base = torch.zeros(world + 1, dtype=torch.int64)
    src_base[1:] = torch.cumsum(recv_counts.sum(1), 0)
    within = torch.zeros(world, mine.numel() + 1, dtype=torch.int64)
    within[:, 1:] = torch.cumsum(recv_counts, 1)
    local_order = []
    for j in range(mine.numel()):
        for s in range(world):
            a = int(src_base[s] + within[s, j])
            local_order.append(torch.arange(a, a + int(recv_counts[s, j]), dtype=torch.int64))
    local_order = torch.cat(local_order) if local_order else torch.zeros(0, dtype=torch.int64)
    local_offsets = torch.zeros(mine.numel() + 1, dtype=torch.int64)
    local_offsets[1:] = torch.cumsum(recv_counts.sum(0), 0)
    return ExchangePlan(owner, mine, send_order, send_splits, recv_counts, recv_splits,
                        local_order, local_offsets)


def dispatch_rows(Xp: torch.Tensor, plan: ExchangePlan, group=None) -> torch.Tensor:
    """Step 3 (and the regrouping of 4): this rank's Xp rows to their experts' owners; returns
    the rows of my experts, expert-major ([local_offsets[-1], ...])."""
    send = Xp.index_select(0, plan.send_order.to(Xp.device))
    recv = Xp.new_empty((int(sum(plan.recv_splits)),) + tuple(Xp.shape[1:]))
    dist.all_to_all_single(recv, send, plan.recv_splits, plan.send_splits, group=group)
    return recv.index_select(0, plan.local_order.to(Xp.device))


def combine_rows(Yp_local: torch.Tensor, plan: ExchangePlan, n_rows: int, group=None) -> torch.Tensor:
    """Step 5: the owner's FFN outputs (expert-major, as dispatch_rows returned the rows) back
    to the ranks they came from; returns this rank's n_rows outputs in its Xp order."""
    dev = Yp_local.device
    recv_order = torch.empty_like(Yp_local)
    recv_order.index_copy_(0, plan.local_order.to(dev), Yp_local)
    back = Yp_local.new_empty((int(sum(plan.send_splits)),) + tuple(Yp_local.shape[1:]))
    dist.all_to_all_single(back, recv_order, plan.send_splits, plan.recv_splits, group=group)
    out = Yp_local.new_zeros((n_rows,) + tuple(Yp_local.shape[1:]))
    out.index_copy_(0, plan.send_order.to(dev), back)
    return out
