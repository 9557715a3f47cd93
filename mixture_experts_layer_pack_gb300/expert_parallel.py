"""Expert-parallel dispatch and combine: the token-row exchange around the experts.

The pages run the layer expert-parallel -- EP16 for the Proxy model, EP64 for
DSv4-Pro ("feat(moe): add a megakernel backend with MOK integration",
Validation) -- the backend takes an expert-parallel process group
("core.transformer.moe.megakernel.mok.backend", MoKMegakernel: ep_group), and
dispatch and combine are the steps on either side of the experts (same PR,
Summary). Here each rank of the group holds its own tokens and owns a
contiguous range of the routed experts; the shared expert stays with the tokens.

This module is the exchange and nothing else:

* ``ExpertPartition``: which rank owns which experts;
* ``make_plan``: from a rank's routing (top-k ids, -1 for a missing route) the
  order of its outgoing rows -- by expert, then token, which is also by owner
  rank because the ranges are contiguous and ascending -- the rows it sends to
  and receives from every rank (one all-to-all of per-expert counts), and the
  permutation that puts the received rows into expert order (expert, then
  source rank, then the source's token order);
* ``dispatch`` / ``return_rows``: the all-to-all(v) of token rows (or of one
  value per row) to the experts' owners and back.

Forward: dispatch x rows (and each route's prob) to the owners, run the local
experts there, return their outputs, combine on the token side. Backward:
dispatch grad_out rows the same way, the owners compute dgrad and accumulate
their experts' weight gradients, return dx rows and the per-route dprob.
The experts, the shared expert and the sums are the caller's (``ep_forward`` /
``ep_backward`` take them as functions), so the exchange runs the same with
NCCL on GPUs or gloo on CPU ranks. On a GPU the owner's experts are the
library's own routed-only step: a ``MoELayer(..., num_experts=len(local),
topk=1, shared_expert=False)`` run with ``forward_topk`` on the received rows
(ids = local expert, probs = the route's prob) returns the prob-weighted
expert outputs, and its ``backward`` the rows' dx, the per-route dprob and the
local experts' main_grad accumulation. The collectives move every row through the
receiving rank's own memory: nothing reads a peer's memory directly.
"""
from __future__ import annotations

import dataclasses

import torch
import torch.distributed as dist


class ExpertPartition:
    """Contiguous ranges of the E routed experts over W ranks: rank r owns
    experts [first[r], first[r + 1]); the first E mod W ranks own one more."""

    def __init__(self, num_experts: int, world: int):
        if world < 1 or num_experts < world:
            raise ValueError("every rank must own at least one expert")
        base, extra = divmod(num_experts, world)
        self.num_experts = num_experts
        self.world = world
        self.first = [r * base + min(r, extra) for r in range(world + 1)]

    def owner(self, e: int) -> int:
        for r in range(self.world):
            if e < self.first[r + 1]:
                return r
        raise ValueError(e)

    def local(self, rank: int) -> range:
        return range(self.first[rank], self.first[rank + 1])

    def owners(self) -> torch.Tensor:
        """owner rank of every expert, [E] int64"""
        return torch.repeat_interleave(torch.arange(self.world),
                                       torch.tensor([self.first[r + 1] - self.first[r] for r in range(self.world)]))


@dataclasses.dataclass
class ExchangePlan:
    perm_src: torch.Tensor      # [R] token of each outgoing row (order: expert, token)
    perm_slot: torch.Tensor     # [R] its slot
    row_of: torch.Tensor        # [T, k] outgoing row of each slot, -1 for a missing route
    counts: torch.Tensor        # [E] outgoing rows per expert
    send_counts: list           # rows to each rank
    recv_counts: list           # rows from each rank
    recv_expert_counts: torch.Tensor  # [W, n_local] rows from each rank per local expert
    local_counts: torch.Tensor  # [n_local] received rows per local expert
    to_expert_order: torch.Tensor  # [n_recv]: received row (source order) at each expert-order position
    local_experts: range


def make_plan(ids: torch.Tensor, part: ExpertPartition, group=None) -> ExchangePlan:
    """The exchange plan of this rank's routing ``ids`` [T, k] (int, -1 = missing).
    One all-to-all of per-expert counts tells every rank what it receives."""
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    if world != part.world:
        raise ValueError("the partition is for another group size")
    ids = ids.to(torch.int64).cpu()
    T, k = ids.shape
    valid = ids >= 0
    flat = torch.nonzero(valid.reshape(-1), as_tuple=False).reshape(-1)   # slot index t * k + s, ascending
    e_of = ids.reshape(-1)[flat]
    order = torch.argsort(e_of, stable=True)         # by expert; within an expert by token (flat is ascending)
    sel = flat[order]
    perm_src, perm_slot = sel // k, sel % k
    row_of = torch.full((T * k,), -1, dtype=torch.int64)
    row_of[sel] = torch.arange(sel.numel())
    counts = torch.bincount(e_of, minlength=part.num_experts)
    send_counts = [int(counts[part.first[d]:part.first[d + 1]].sum()) for d in range(world)]
    # per-expert counts to each owner: the owner learns how many rows of each of its
    # experts every rank sends
    n_local = len(part.local(rank))
    sizes_out = [part.first[d + 1] - part.first[d] for d in range(world)]
    recv = torch.empty(world * n_local, dtype=torch.int64)
    dist.all_to_all_single(recv, counts.clone(), [n_local] * world, sizes_out, group=group)
    recv_expert_counts = recv.reshape(world, n_local)
    recv_counts = [int(x) for x in recv_expert_counts.sum(1)]
    local_counts = recv_expert_counts.sum(0)
    # received rows arrive by source rank, each source's block by expert; expert order
    # takes, for each local expert, its rows from source 0, 1, ...
    src_base = torch.cumsum(torch.tensor([0] + recv_counts[:-1]), 0)
    within = torch.cumsum(torch.cat([torch.zeros(world, 1, dtype=torch.int64), recv_expert_counts[:, :-1]], 1), 1)
    pieces = []
    for j in range(n_local):
        for s in range(world):
            start = int(src_base[s] + within[s, j])
            pieces.append(torch.arange(start, start + int(recv_expert_counts[s, j])))
    to_expert_order = torch.cat(pieces) if pieces else torch.zeros(0, dtype=torch.int64)
    return ExchangePlan(perm_src, perm_slot, row_of.reshape(T, k), counts, send_counts, recv_counts,
                        recv_expert_counts, local_counts, to_expert_order, part.local(rank))


def dispatch(plan: ExchangePlan, rows: torch.Tensor, group=None) -> torch.Tensor:
    """Token-side rows [R, ...] in outgoing order to their experts' owners;
    returns the received rows in expert order."""
    recv = rows.new_empty((sum(plan.recv_counts),) + tuple(rows.shape[1:]))
    dist.all_to_all_single(recv, rows.contiguous(), plan.recv_counts, plan.send_counts, group=group)
    return recv[plan.to_expert_order.to(recv.device)]


def return_rows(plan: ExchangePlan, rows: torch.Tensor, group=None) -> torch.Tensor:
    """Owner-side rows [n_recv, ...] in expert order back to the token side;
    returns them in the outgoing order of ``plan``."""
    src_order = torch.empty_like(rows)
    src_order[plan.to_expert_order.to(rows.device)] = rows
    back = rows.new_empty((sum(plan.send_counts),) + tuple(rows.shape[1:]))
    dist.all_to_all_single(back, src_order.contiguous(), plan.send_counts, plan.recv_counts, group=group)
    return back


def ep_forward(hidden, ids, pp, part, experts_fwd, shared_fwd, combine, group=None):
    """Expert-parallel forward of this rank's tokens.

    ids, pp [T, k]: the routing (fixed width, -1 = missing); experts_fwd(rows,
    local_counts, probs) -> (outputs, cache) runs this rank's experts on their
    received rows (expert order); shared_fwd(hidden) -> shared output;
    combine(shared_out, routed_rows, row_of, pp) -> out. Returns (out, state)."""
    plan = make_plan(ids, part, group)
    x_rows = dispatch(plan, hidden[plan.perm_src], group)
    p_rows = dispatch(plan, pp[plan.perm_src, plan.perm_slot], group)
    y_rows, cache = experts_fwd(x_rows, plan.local_counts, p_rows)
    y_back = return_rows(plan, y_rows, group)
    out = combine(shared_fwd(hidden), y_back, plan.row_of, pp)
    return out, dict(plan=plan, x_rows=x_rows, p_rows=p_rows, cache=cache)


def ep_backward(grad_out, state, experts_bwd, shared_bwd, unpermute, group=None):
    """Expert-parallel backward: grad_out rows to the owners, experts_bwd(x_rows,
    go_rows, probs, local_counts, cache) -> (dx_rows, dprob_rows) there (it
    accumulates the local experts' weight gradients), dx rows and per-route
    dprobs back; unpermute(shared_dx, dx_back, dprob_back, plan) -> (dhidden,
    dprobs) on the token side."""
    plan = state["plan"]
    go_rows = dispatch(plan, grad_out[plan.perm_src], group)
    dx_rows, dprob_rows = experts_bwd(state["x_rows"], go_rows, state["p_rows"], plan.local_counts, state["cache"])
    dx_back = return_rows(plan, dx_rows, group)
    dprob_back = return_rows(plan, dprob_rows, group)
    return unpermute(shared_bwd(grad_out), dx_back, dprob_back, plan)
