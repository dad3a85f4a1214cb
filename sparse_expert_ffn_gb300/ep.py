"""Expert parallelism: the experts of one MoE layer split across the ranks of
a process group (one GPU each, one machine), token rows exchanged with
all-to-all collectives.

cf-1.com section 4.1 (GPU-to-GPU bandwidth for the communication between
experts on several cards) and section 4.3 (several GPUs of one machine).
Rank g owns experts [g*E/G, (g+1)*E/G).  One forward on every rank, for that
rank's own tokens:

  1. route its tokens with the full router and gather the rows into expert
     order (colibri_route_static, colibri_gather_rows): the rows bound for
     owner g are the contiguous range of g's experts;
  2. exchange the per-expert counts (all-to-all of a [G, E/G] table), then
     the rows (all-to-all with those row counts as split sizes);
  3. run the owned experts on the rows received (colibri_forward_routed on a
     handle that holds only them, one expert per row, gate 1), the rows of
     each source in that source's expert order;
  4. send the results back with the reverse all-to-all; they land in the
     sender's expert order, where the gate-weighted combine (colibri_
     combine_rows, j in order, float32) reads them.

The exchange is this module's part (torch.distributed as the collective
library, NCCL on GPUs); every step on the data runs in the library's
kernels.  The steps are injectable callables, so that the exchange logic can
be run on CPU tensors with the gloo backend against a reference."""

from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Optional

import torch


@dataclass
class ExchangePlan:
    """Row counts of one exchange, from the source's per-expert pair counts.

    send_rows[g]: rows this rank sends to owner g (a contiguous range of its
    expert-ordered rows); send_table[g, e]: of those, rows of g's local
    expert e.  After the counts are exchanged, recv_table[s, e]: rows source s
    sends for this rank's local expert e, recv_rows[s] their sum."""

    world: int
    experts_per_rank: int
    send_table: torch.Tensor          # [G, E/G] int64
    recv_table: Optional[torch.Tensor] = None

    @staticmethod
    def from_counts(counts: torch.Tensor, world: int) -> "ExchangePlan":
        counts = counts.to(torch.int64).cpu()
        E = counts.numel()
        if E % world:
            raise ValueError(f"{E} experts do not split evenly over {world} ranks")
        return ExchangePlan(world, E // world, counts.view(world, E // world).clone())

    @property
    def send_rows(self) -> List[int]:
        return self.send_table.sum(dim=1).tolist()

    @property
    def recv_rows(self) -> List[int]:
        assert self.recv_table is not None, "exchange the counts first"
        return self.recv_table.sum(dim=1).tolist()

    def local_expert_ids(self) -> torch.Tensor:
        """Local expert id of every received row, in arrival order (sources in
        rank order, inside each source its expert order)."""
        assert self.recv_table is not None, "exchange the counts first"
        ids = torch.arange(self.experts_per_rank, dtype=torch.int32)
        return torch.cat([torch.repeat_interleave(ids, self.recv_table[s])
                          for s in range(self.world)])


def exchange_counts(plan: ExchangePlan, group=None, device="cpu") -> ExchangePlan:
    """All-to-all of the [G, E/G] count table: row g goes to rank g."""
    import torch.distributed as dist
    send = plan.send_table.to(device)
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send, group=group)
    plan.recv_table = recv.cpu()
    return plan


def exchange_rows(rows: torch.Tensor, send_rows: List[int], recv_rows: List[int],
                  group=None) -> torch.Tensor:
    """All-to-all of row blocks: send_rows[g] consecutive rows to rank g,
    recv_rows[s] rows arriving from rank s, in rank order."""
    import torch.distributed as dist
    out = rows.new_empty((sum(recv_rows),) + tuple(rows.shape[1:]))
    dist.all_to_all_single(out, rows.contiguous(), output_split_sizes=recv_rows,
                           input_split_sizes=send_rows, group=group)
    return out


@dataclass
class Steps:
    """The data steps of one forward (library kernels by default).

    route(x) -> (topk_idx [T, k] int32, topk_w [T, k] float32, counts [E] int32, perm [T*k] int32)
    gather(x, perm, k) -> rows [T*k, d] in expert order
    experts(rows, local_ids) -> out rows [R, d], out[r] = FFN_{local_ids[r]}(rows[r])
    combine(back, topk_w, perm) -> y [T, d]"""

    route: Callable
    gather: Callable
    experts: Callable
    combine: Callable


def ep_forward(x: torch.Tensor, steps: Steps, world: int, group=None,
               count_device="cpu") -> torch.Tensor:
    """One expert-parallel forward of this rank's tokens x [T, d]."""
    topk_idx, topk_w, counts, perm = steps.route(x)
    k = topk_idx.shape[1]
    rows = steps.gather(x, perm, k)
    plan = exchange_counts(ExchangePlan.from_counts(counts, world), group, count_device)
    recv = exchange_rows(rows, plan.send_rows, plan.recv_rows, group)
    out = steps.experts(recv, plan.local_expert_ids().to(recv.device))
    back = exchange_rows(out, plan.recv_rows, plan.send_rows, group)
    return steps.combine(back, topk_w, perm)


class ExpertParallelLayer:
    """One rank's share of an expert-parallel layer on its GPU: the full
    router (replicated) and a handle over its E/G experts.

    w_router [d, E], router_bias [E] or None; w_gate, w_up [E/G, d, f] and
    w_down [E/G, f, d]: this rank's experts.  max_tokens bounds T per forward
    on every rank (an owner may receive up to world * max_tokens * top_k
    rows).  `world` defaults to the size of `group` (1 without a process
    group); the data steps (route, gather, experts, combine) are methods, so
    that several ranks' shares can also be driven from one process."""

    def __init__(self, w_router, router_bias, w_gate, w_up, w_down, top_k: int, n_experts: int,
                 max_tokens: int, group=None, world: Optional[int] = None):
        import torch.distributed as dist
        from . import DTYPE_BF16, DTYPE_FP32, MoELayer
        self.group = group
        if world is None:
            world = dist.get_world_size(group) if dist.is_initialized() else 1
        self.world = world
        self.E, self.k = n_experts, top_k
        self.El = n_experts // self.world
        if self.El * self.world != n_experts or w_gate.shape[0] != self.El:
            raise ValueError("each rank holds n_experts / world experts")
        dev = w_router.device
        self.d = w_router.shape[0]
        self.dtype = w_router.dtype
        self.w_router = w_router.contiguous()
        self.bias = None if router_bias is None else router_bias.to(dev, torch.float32).contiguous()
        # the owned experts; their router is never run (routing is the caller's)
        zero_router = torch.zeros(self.d, self.El, dtype=self.dtype, device=dev)
        self.owner = MoELayer(zero_router, w_gate, w_up, w_down, 1,
                              max_tokens=self.world * max_tokens * top_k)
        self._dt = DTYPE_BF16 if self.dtype == torch.bfloat16 else DTYPE_FP32
        T, k = max_tokens, top_k
        self._idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        self._w = torch.empty((T, k), dtype=torch.float32, device=dev)
        self._cnt = torch.empty((n_experts,), dtype=torch.int32, device=dev)
        self._perm = torch.empty((T * k,), dtype=torch.int32, device=dev)
        self._inv = torch.empty((T * k,), dtype=torch.int32, device=dev)
        self.max_tokens = max_tokens

    @staticmethod
    def _check(st, what):
        from . import ColibriError
        if st != 0:
            raise ColibriError(st, what)

    def route(self, x):
        """(topk_idx [T, k], topk_w [T, k], counts [E], perm [T*k]) of x [T, d]
        (colibri_route_static); an empty batch has all counts 0."""
        from . import library
        T = x.shape[0]
        if T == 0:
            self._cnt.zero_()
        else:
            s = torch.cuda.current_stream().cuda_stream
            st = library().colibri_route_static(
                x.data_ptr(), self.w_router.data_ptr(),
                None if self.bias is None else self.bias.data_ptr(), T, self.d, self.E, self.k,
                self._dt, self._idx.data_ptr(), self._w.data_ptr(), self._cnt.data_ptr(),
                self._perm.data_ptr(), s)
            self._check(st, "colibri_route_static")
        return self._idx[:T], self._w[:T], self._cnt, self._perm[:T * self.k]

    def gather(self, x, perm, k):
        """x's rows in the expert order of perm (colibri_gather_rows)."""
        from . import library
        rows = torch.empty((perm.numel(), self.d), dtype=x.dtype, device=x.device)
        if perm.numel():
            s = torch.cuda.current_stream().cuda_stream
            self._check(library().colibri_gather_rows(
                x.data_ptr(), x.shape[0], perm.data_ptr(), k, perm.numel(), self.d, self._dt,
                rows.data_ptr(), s), "colibri_gather_rows")
        return rows

    def experts(self, rows, ids):
        """out[r] = FFN_{ids[r]}(rows[r]) over this rank's experts
        (colibri_forward_routed, one expert per row, gate 1)."""
        if rows.shape[0] == 0:
            return torch.empty_like(rows)
        ones = torch.ones(rows.shape[0], dtype=torch.float32, device=rows.device)
        return self.owner.forward_routed(rows, ids.to(torch.int32).contiguous(), ones)

    def combine(self, back, topk_w, perm):
        """y [T, d]: the gate-weighted sum of each token's rows of `back`
        (expert order of perm) (colibri_combine_rows)."""
        from . import library
        T = topk_w.shape[0]
        y = torch.empty((T, self.d), dtype=self.dtype, device=back.device)
        if T:
            s = torch.cuda.current_stream().cuda_stream
            self._check(library().colibri_combine_rows(
                back.data_ptr(), self._dt, topk_w.data_ptr(), perm.data_ptr(), T, self.k, self.d,
                self._dt, self._inv.data_ptr(), y.data_ptr(), s), "colibri_combine_rows")
        return y

    def steps(self) -> Steps:
        return Steps(self.route, self.gather, self.experts, self.combine)

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.shape[0] > self.max_tokens:
            raise ValueError("more tokens than max_tokens")
        return ep_forward(x.contiguous(), self.steps(), self.world, self.group, count_device=x.device)

    def check(self) -> int:
        return self.owner.check()

    def close(self):
        self.owner.close()
