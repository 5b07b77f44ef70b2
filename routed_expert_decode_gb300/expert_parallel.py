"""Expert-parallel split of the routed-MoE layer, one rank per GPU.

The routed experts are partitioned into contiguous ranges, one per rank; the
shared expert is held by every rank and computed once per token.  This is the
multi-GPU expert residency the pages name as the next lever once one GPU's
memory or bandwidth is the limit (NeutronStar README, next-levers paragraph;
the two-worker split of NeutronStar glm-local README, "Roadmap").

Two schedules:

* ``decode`` -- every rank holds the same T tokens (single-token decode,
  speculative-verify batches).  Each rank computes its own experts for every
  token with ``moe_layer_experts`` (rank 0 adds the shared expert); one sum
  all-reduce of y [T, d] fp32 gives the layer.
* ``prefill`` -- each rank holds its own tokens.  Each rank routes them and
  sends every row that names an expert of rank r -- its x and its router
  logits, from which r recomputes the same routing -- to r in one all-to-all;
  the owners run ``moe_layer_experts`` on the rows they received and a second
  all-to-all returns the partial outputs, which each rank adds, in rank order,
  to its own shared-expert output.

Only host logic lives here: the per-rank compute is a function handed to the
class (``for_layer`` binds the library's ``moe_layer_experts`` and
``moe_route``), so the partition and the exchanges also run on CPU ranks
(gloo) with any compute function.  The sum of the ranks' partial outputs is
the layer up to fp32 summation order (shared first, then each rank's experts
in slot order), within the layer's output tolerance.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Tuple

import torch
import torch.distributed as dist


def expert_ranges(n_expert: int, world: int) -> List[Tuple[int, int]]:
    """Contiguous, balanced expert ranges [lo, hi) of ranks 0..world-1."""
    if world < 1 or n_expert < world:
        raise ValueError(f"cannot split {n_expert} experts over {world} ranks")
    return [(r * n_expert // world, (r + 1) * n_expert // world) for r in range(world)]


def owner_of(expert: int, ranges: List[Tuple[int, int]]) -> int:
    for r, (lo, hi) in enumerate(ranges):
        if lo <= expert < hi:
            return r
    raise ValueError(f"expert {expert} outside every range")


# partial(x [rows, d], logits [rows, E], lo, hi, with_shared) -> y [rows, d] fp32
PartialFn = Callable[[torch.Tensor, torch.Tensor, int, int, bool], torch.Tensor]
# route(logits [rows, E]) -> expert indices [rows, top_k] (int)
RouteFn = Callable[[torch.Tensor], torch.Tensor]


class ExpertParallel:
    """One rank's view of an expert-parallel layer."""

    def __init__(self, n_expert: int, rank: int, world: int, partial: PartialFn,
                 route: Optional[RouteFn] = None, group=None):
        self.n_expert, self.rank, self.world = n_expert, rank, world
        self.ranges = expert_ranges(n_expert, world)
        self.lo, self.hi = self.ranges[rank]
        self.partial = partial
        self.route = route
        self.group = group

    # ------------------------------------------------------------------ decode
    def decode(self, x: torch.Tensor, logits: torch.Tensor) -> torch.Tensor:
        """Every rank passes the same tokens; every rank returns the layer's y."""
        y = self.partial(x, logits, self.lo, self.hi, self.rank == 0)
        if self.world > 1:
            dist.all_reduce(y, op=dist.ReduceOp.SUM, group=self.group)
        return y

    # ------------------------------------------------------------------ prefill
    def dispatch_plan(self, idx: torch.Tensor) -> List[torch.Tensor]:
        """Row indices of this rank's tokens to send to each rank: the rows that
        name at least one of that rank's experts, in token order."""
        out = []
        for lo, hi in self.ranges:
            hit = ((idx >= lo) & (idx < hi)).any(dim=1)
            out.append(torch.nonzero(hit, as_tuple=False).flatten())
        return out

    def prefill(self, x: torch.Tensor, logits: torch.Tensor) -> torch.Tensor:
        """Each rank passes its own tokens and gets its own tokens' y back."""
        if self.route is None:
            raise ValueError("prefill needs a route function")
        dev = x.device
        d, E = x.shape[1], logits.shape[1]
        sel = self.dispatch_plan(self.route(logits))
        send_n = torch.tensor([len(s) for s in sel], dtype=torch.int64)
        recv_n = torch.empty_like(send_n)
        if self.world > 1:
            # the counts travel on the collective's own device
            sn, rn = send_n.to(dev), torch.empty(self.world, dtype=torch.int64, device=dev)
            dist.all_to_all_single(rn, sn, group=self.group)
            recv_n = rn.cpu()
        else:
            recv_n = send_n.clone()
        order = torch.cat(sel) if sel else torch.empty(0, dtype=torch.long, device=dev)
        send_x, send_l = x.index_select(0, order), logits.index_select(0, order)
        s_split, r_split = send_n.tolist(), recv_n.tolist()
        recv_x = torch.empty((sum(r_split), d), dtype=x.dtype, device=dev)
        recv_l = torch.empty((sum(r_split), E), dtype=logits.dtype, device=dev)
        self._exchange(recv_x, send_x, r_split, s_split)
        self._exchange(recv_l, send_l, r_split, s_split)
        # the owner's share of the rows it received (no shared expert: each
        # token's own rank adds that)
        if recv_x.shape[0]:
            y_recv = self.partial(recv_x, recv_l, self.lo, self.hi, False)
        else:
            y_recv = torch.empty((0, d), dtype=torch.float32, device=dev)
        y_back = torch.empty((sum(s_split), d), dtype=torch.float32, device=dev)
        self._exchange(y_back, y_recv, s_split, r_split)
        # this rank's tokens: shared expert, then the owners' partials in rank order
        y = self.partial(x, logits, 0, 0, True)
        start = 0
        for s in sel:
            n = len(s)
            if n:
                y.index_add_(0, s, y_back[start:start + n])
            start += n
        return y

    def _exchange(self, out: torch.Tensor, inp: torch.Tensor, out_split, in_split):
        if self.world > 1:
            dist.all_to_all_single(out, inp.contiguous(), out_split, in_split, group=self.group)
        else:
            out.copy_(inp)

    # ------------------------------------------------------------------ GPU binding
    @classmethod
    def for_layer(cls, layer, bias: torch.Tensor, rank: int, world: int, group=None,
                  weights=None) -> "ExpertParallel":
        """Bind a resident ``moe.Layer`` (weights of at least this rank's experts,
        e.g. through an expert -> slot table in ``weights``) to the schedules:
        ``moe_layer_experts`` computes, ``moe_route`` routes."""
        from . import moe

        wts = weights if weights is not None else layer.weights
        desc = layer.desc()

        def partial(x, logits, lo, hi, with_shared):
            T = x.shape[0]
            y = torch.empty((T, layer.d), dtype=torch.float32, device=x.device)
            ws = layer.workspace(T, 0)
            moe.layer_experts(desc, wts, x.contiguous(), logits.contiguous(), bias, y, ws, lo,
                              hi, with_shared)
            return y

        def route(logits):
            T = logits.shape[0]
            dev = logits.device
            idx = torch.empty((T, layer.top_k), dtype=torch.int32, device=dev)
            w = torch.empty((T, layer.top_k), dtype=torch.float32, device=dev)
            off = torch.empty(layer.n_expert + 1, dtype=torch.int32, device=dev)
            perm = torch.empty(T * layer.top_k, dtype=torch.int32, device=dev)
            pos = torch.empty(T * layer.top_k, dtype=torch.int32, device=dev)
            moe.route(desc, logits.contiguous(), bias, idx, w, off, perm, pos)
            return idx

        return cls(layer.n_expert, rank, world, partial, route, group)
