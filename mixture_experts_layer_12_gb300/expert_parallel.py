"""Expert parallelism: the experts are split over G ranks (one GPU each), the
dispatched token rows travel to the rank that owns their expert and the
expert outputs travel back before the combine.

This is the all-to-all expert-parallel scheme of the CANN ops-transformer
MoE article, section 3 (communication: all-to-all of the tokens grouped by
destination expert), on top of the library's own steps:

  rank r holds experts [r*El, (r+1)*El), El = E / G, and its own tokens;
  1. moe_route on its tokens (all E experts: the router weights are
     replicated), then moe_dispatch_rows -- the kept rows in dispatch order,
     which is expert-major, so the rows bound for rank d are one contiguous
     slice: offsets[d*El] .. offsets[(d+1)*El];
  2. all-to-all of the per-expert row counts (each destination receives the
     El counts of its experts from every source), then of the rows;
  3. the received rows arrive grouped by source, then by local expert:
     moe_expert_ffn runs on them as they are, with G*El segments (segment i
     = source i // El, local expert i % El);
  4. the outputs, in that same order, go back by the reverse all-to-all and
     land in the source's dispatch order; moe_combine finishes.

Capacity drops are decided per rank over its own tokens (as in a replica of
the whole layer), so every rank's y equals the single-GPU layer's y on the
same tokens.  The exchange is an object with `counts` and `rows` methods
(TorchExchange: torch.distributed all_to_all_single, NCCL on GPUs, gloo on
CPU ranks); the compute steps are the library's C-ABI calls (CudaOps).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import (MOE_GATE_TOPK_SOFTMAX, alloc_route_workspace, alloc_routing, alloc_workspace,
               make_shape, moe_combine, moe_dispatch_rows, moe_expert_ffn, moe_route)


def send_splits(offsets: list[int], world: int) -> list[int]:
    """Rows of the dispatch order bound for each rank (E divisible by world)."""
    E = len(offsets) - 1
    el = E // world
    return [offsets[(d + 1) * el] - offsets[d * el] for d in range(world)]


def segment_offsets(recv_counts: torch.Tensor) -> list[int]:
    """Row offsets of the G*El segments of a received buffer: recv_counts
    [G, El] holds the rows of local expert e received from source s."""
    out = [0]
    for n in recv_counts.reshape(-1).tolist():
        out.append(out[-1] + int(n))
    return out


class TorchExchange:
    """All-to-all over a torch.distributed process group."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)

    def counts(self, send: torch.Tensor) -> torch.Tensor:
        """send [G, El] int64 (row d: counts for rank d's experts) -> [G, El]
        (row s: counts source s sends for this rank's experts)."""
        recv = torch.empty_like(send)
        self.dist.all_to_all_single(recv, send.contiguous(), group=self.group)
        return recv

    def rows(self, send: torch.Tensor, send_split: list[int], recv_split: list[int]) -> torch.Tensor:
        recv = send.new_empty((sum(recv_split),) + tuple(send.shape[1:]))
        self.dist.all_to_all_single(recv, send.contiguous(), recv_split, send_split,
                                    group=self.group)
        return recv


@dataclass
class Routed:
    """One rank's routing and the rows it sends."""
    T: int
    ids: torch.Tensor
    weights: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    perm: torch.Tensor
    slot: torch.Tensor
    rows: torch.Tensor          # [kept, H] kept token rows in dispatch order
    send_split: list[int]       # rows to each rank
    send_counts: torch.Tensor   # [G, El] int64 (CPU)


class CudaOps:
    """The compute steps on this rank's GPU through the C ABI."""

    def __init__(self, w_router, w1_local, w2_local, k, E, bias=None, capacity_factor=None,
                 gating=MOE_GATE_TOPK_SOFTMAX, act="gelu"):
        self.w_router, self.w1, self.w2, self.bias = w_router, w1_local, w2_local, bias
        self.k, self.E = int(k), int(E)
        self.El, self.F, self.H = w2_local.shape[0], w2_local.shape[1], w2_local.shape[2]
        self.cf, self.gating, self.act = capacity_factor, int(gating), act

    def _shape(self, T):
        return make_shape(T, self.H, self.F, self.E, self.k, self.cf, self.gating, self.act)

    def route(self, x):
        T = x.shape[0]
        s = self._shape(T)
        r = alloc_routing(T, self.E, self.k, x.device)
        ws = alloc_route_workspace(s, x.device)
        moe_route(s, x, self.w_router, self.bias, r.ids, r.weights, r.counts, r.offsets, r.perm,
                  r.slot, ws)
        return r

    def dispatch_rows(self, x, r):
        xp = torch.empty(x.shape[0] * self.k, self.H, dtype=x.dtype, device=x.device)
        moe_dispatch_rows(self._shape(x.shape[0]), x, r.perm, r.offsets, xp)
        return xp

    def expert_ffn(self, rows, seg_offsets: list[int]):
        n = rows.shape[0]
        Y = torch.empty_like(rows)
        if n == 0:
            return Y
        s = make_shape(n, self.H, self.F, self.El, 1, None, MOE_GATE_TOPK_SOFTMAX, self.act)
        ws = alloc_workspace(s, rows.device)
        so = torch.tensor(seg_offsets, dtype=torch.int32, device=rows.device)
        moe_expert_ffn(s, len(seg_offsets) - 1, rows, self.w1, self.w2, so, Y, ws)
        return Y

    def combine(self, Y, r, T):
        y = torch.empty(T, self.H, dtype=Y.dtype, device=Y.device)
        moe_combine(self._shape(T), Y, r.weights, r.slot, y)
        return y


class ExpertParallelMoE:
    """One rank of an expert-parallel MoE layer (E experts over `world`
    ranks; this rank holds experts [rank*E/world, (rank+1)*E/world))."""

    def __init__(self, ops, rank: int, world: int, exchange=None):
        if ops.E % world:
            raise ValueError(f"E = {ops.E} experts do not split over {world} ranks")
        self.ops, self.rank, self.world, self.exchange = ops, rank, world, exchange
        self.El = ops.E // world

    # -- the three local phases (the exchange happens between them) --------

    def send(self, x) -> Routed:
        r = self.ops.route(x)
        offsets = [int(v) for v in r.offsets.cpu().tolist()]
        xp = self.ops.dispatch_rows(x, r)
        counts = r.counts.cpu().to(torch.int64).reshape(self.world, self.El)
        return Routed(x.shape[0], r.ids, r.weights, r.counts, r.offsets, r.perm, r.slot,
                      xp[: offsets[-1]], send_splits(offsets, self.world), counts)

    def compute(self, recv_rows, recv_counts: torch.Tensor):
        """Expert FFN of the rows received from every source ([G, El] counts)."""
        return self.ops.expert_ffn(recv_rows, segment_offsets(recv_counts))

    def finish(self, routed: Routed, Y_back):
        """Combine this rank's tokens from its expert outputs (dispatch order)."""
        full = Y_back.new_zeros((routed.T * self.ops.k,) + tuple(Y_back.shape[1:]))
        full[: Y_back.shape[0]] = Y_back
        return self.ops.combine(full, routed, routed.T)

    # -- the whole layer -------------------------------------------------------

    def forward(self, x):
        routed = self.send(x)
        recv_counts = self.exchange.counts(routed.send_counts)
        recv_split = [int(v) for v in recv_counts.sum(dim=1).tolist()]
        recv_rows = self.exchange.rows(routed.rows, routed.send_split, recv_split)
        Y = self.compute(recv_rows, recv_counts)
        Y_back = self.exchange.rows(Y, recv_split, routed.send_split)
        return self.finish(routed, Y_back)
