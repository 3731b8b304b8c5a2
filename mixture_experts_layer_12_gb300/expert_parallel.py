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
     moe_expert_ffn runs on them with G*El segments (segment i = source
     i // El, local expert i % El);
  4. the outputs go back by the reverse all-to-all, are put back in the
     source's dispatch order, and moe_combine finishes.

Capacity drops are decided per rank over its own tokens (as in a replica of
the whole layer), so every rank's y equals the single-GPU layer's y on the
same tokens.

Two exchange modes:
  * padded=False (default): the row all-to-alls carry exactly the rows; their
    split sizes are read to the host once per step, right after the count
    exchange (one small device-to-host copy -- the step's only host
    synchronisation).
  * padded=True: every (source, destination) block of the row all-to-alls
    has room for the most rows a source can send one destination (T*k, or
    El * capacity with a capacity factor), so the exchanges have equal
    splits and every index step runs on the device: nothing is read back
    before the combine and the step can be captured in a CUDA graph.  The
    price is G times the exchanged bytes, and a receive buffer and expert
    workspace for G*T*k rows -- meant for small batches (decode steps).
Buffers are allocated once per batch size and reused.

The exchange is an object with `counts`, `rows` and `rows_even` methods
(TorchExchange: torch.distributed all_to_all_single, NCCL on GPUs, gloo on
CPU ranks); the compute steps are the library's C-ABI calls (CudaOps).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import (MOE_GATE_TOPK_SOFTMAX, alloc_route_workspace, alloc_routing, alloc_workspace,
               make_shape, moe_combine, moe_dispatch_rows, moe_expert_capacity, moe_expert_ffn,
               moe_route)


def send_splits(offsets: list[int], world: int) -> list[int]:
    """Rows of the dispatch order bound for each rank (E divisible by world)."""
    E = len(offsets) - 1
    el = E // world
    return [offsets[(d + 1) * el] - offsets[d * el] for d in range(world)]


def segment_offsets(recv_counts: torch.Tensor) -> torch.Tensor:
    """Row offsets [G*El + 1] (int32, on recv_counts' device) of the G*El
    segments of a received buffer: recv_counts [G, El] holds the rows of
    local expert e received from source s, sources in order."""
    flat = recv_counts.reshape(-1).to(torch.int32)
    out = torch.zeros(flat.numel() + 1, dtype=torch.int32, device=flat.device)
    torch.cumsum(flat, 0, out=out[1:])
    return out


class TorchExchange:
    """All-to-all over a torch.distributed process group."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)

    def counts(self, send: torch.Tensor) -> torch.Tensor:
        """send [G, El] (row d: counts for rank d's experts) -> [G, El]
        (row s: counts source s sends for this rank's experts)."""
        recv = torch.empty_like(send)
        self.dist.all_to_all_single(recv, send.contiguous(), group=self.group)
        return recv

    def rows(self, send: torch.Tensor, send_split: list[int], recv_split: list[int],
             out: torch.Tensor | None = None) -> torch.Tensor:
        recv = out if out is not None else send.new_empty((sum(recv_split),) + tuple(send.shape[1:]))
        self.dist.all_to_all_single(recv, send.contiguous(), recv_split, send_split,
                                    group=self.group)
        return recv

    def rows_even(self, send: torch.Tensor, out: torch.Tensor) -> torch.Tensor:
        """Equal splits: block d of `send` goes to rank d, block s of `out`
        comes from rank s."""
        self.dist.all_to_all_single(out, send.contiguous(), group=self.group)
        return out


@dataclass
class Routed:
    """One rank's routing and what it sends."""
    T: int
    ids: torch.Tensor
    weights: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    perm: torch.Tensor
    slot: torch.Tensor
    send_counts: torch.Tensor   # [G, El] kept rows per destination expert (device)
    rows: torch.Tensor          # exact: [T*k, H] dispatch order; padded: [G*cap, H] blocks


class CudaOps:
    """The compute steps on this rank's GPU through the C ABI, with every
    buffer allocated once per batch size (`prepare`)."""

    def __init__(self, w_router, w1_local, w2_local, k, E, bias=None, capacity_factor=None,
                 gating=MOE_GATE_TOPK_SOFTMAX, act="gelu"):
        self.w_router, self.w1, self.w2, self.bias = w_router, w1_local, w2_local, bias
        self.k, self.E = int(k), int(E)
        self.El, self.F, self.H = w2_local.shape[0], w2_local.shape[1], w2_local.shape[2]
        self.cf, self.gating, self.act = capacity_factor, int(gating), act
        self.device = w2_local.device
        self._T = None
        self._ffn_rows = 0

    def _shape(self, T):
        return make_shape(T, self.H, self.F, self.E, self.k, self.cf, self.gating, self.act)

    def prepare(self, T: int):
        """Routing buffers, route workspace, dispatch-ordered rows and y for T tokens."""
        if self._T == T:
            return
        s = self._shape(T)
        self.r = alloc_routing(T, self.E, self.k, self.device)
        self.route_ws = alloc_route_workspace(s, self.device)
        self.xp = torch.empty(max(T * self.k, 1), self.H, dtype=torch.bfloat16, device=self.device)
        self.y = torch.empty(T, self.H, dtype=torch.bfloat16, device=self.device)
        self._T = T

    def max_rows_to_one_rank(self, T: int) -> int:
        """The most rows one source can send one destination: all of its T*k
        assignments, or El experts' capacity when a capacity factor is set."""
        c = moe_expert_capacity(self._shape(T))
        return T * self.k if c < 0 else min(T * self.k, self.El * c)

    def route(self, x):
        self.prepare(x.shape[0])
        r = self.r
        moe_route(self._shape(x.shape[0]), x, self.w_router, self.bias, r.ids, r.weights, r.counts,
                  r.offsets, r.perm, r.slot, self.route_ws)
        return r

    def dispatch_rows(self, x, r):
        moe_dispatch_rows(self._shape(x.shape[0]), x, r.perm, r.offsets, self.xp)
        return self.xp

    def expert_ffn(self, rows, seg_offsets: torch.Tensor, n_segments: int):
        """Y[i] = FFN_{segment's expert}(rows[i]); rows [n, H] (n = capacity,
        only rows inside the segments are computed); seg_offsets on device."""
        n = rows.shape[0]
        if n == 0:
            return torch.empty_like(rows)
        if n > self._ffn_rows:  # grow-only: allocated once for the largest row capacity
            s = make_shape(n, self.H, self.F, self.El, 1, None, MOE_GATE_TOPK_SOFTMAX, self.act)
            self.ffn_ws = alloc_workspace(s, rows.device)
            self.ffn_Y = torch.empty(n, self.H, dtype=torch.bfloat16, device=rows.device)
            self._ffn_rows = n
        s = make_shape(n, self.H, self.F, self.El, 1, None, MOE_GATE_TOPK_SOFTMAX, self.act)
        Y = self.ffn_Y[:n]
        moe_expert_ffn(s, n_segments, rows, self.w1, self.w2, seg_offsets, Y, self.ffn_ws)
        return Y

    def combine(self, Y, r, T):
        moe_combine(self._shape(T), Y, r.weights, r.slot, self.y)
        return self.y


class ExpertParallelMoE:
    """One rank of an expert-parallel MoE layer (E experts over `world`
    ranks; this rank holds experts [rank*E/world, (rank+1)*E/world))."""

    def __init__(self, ops, rank: int, world: int, exchange=None, padded: bool = False):
        if ops.E % world:
            raise ValueError(f"E = {ops.E} experts do not split over {world} ranks")
        self.ops, self.rank, self.world, self.exchange = ops, rank, world, exchange
        self.El = ops.E // world
        self.padded = bool(padded)
        self._bufs = {}
        self.cap = None

    def _buf(self, name: str, rows: int, like: torch.Tensor) -> torch.Tensor:
        """A [rows, H] buffer of `like`'s dtype and device, allocated once."""
        b = self._bufs.get(name)
        if b is None or b.shape[0] != rows or b.dtype != like.dtype or b.device != like.device:
            b = torch.zeros((rows,) + tuple(like.shape[1:]), dtype=like.dtype, device=like.device)
            self._bufs[name] = b
        return b

    def _ramp(self, n: int, device) -> torch.Tensor:
        b = self._bufs.get(("ramp", n))
        if b is None or b.device != torch.device(device):
            b = torch.arange(n, device=device)
            self._bufs[("ramp", n)] = b
        return b

    # -- the three local phases (the exchanges happen between them) --------

    def send(self, x) -> Routed:
        """Route this rank's tokens and lay out the rows each rank receives."""
        T = x.shape[0]
        r = self.ops.route(x)
        xp = self.ops.dispatch_rows(x, r)
        counts = r.counts.reshape(self.world, self.El)
        if not self.padded:
            return Routed(T, r.ids, r.weights, r.counts, r.offsets, r.perm, r.slot, counts, xp)
        # block d of the send buffer: the rows bound for rank d (a contiguous
        # slice of the dispatch order), then unused room
        self.cap = cap = max(1, self.ops.max_rows_to_one_rank(T))
        ramp = self._ramp(self.world * cap, xp.device)
        start = r.offsets[:-1].reshape(self.world, self.El)[:, 0].long()
        n_d = counts.sum(dim=1).long()
        d = ramp // cap
        j = ramp - d * cap
        src = torch.where(j < n_d[d], start[d] + j, torch.zeros_like(j))
        send_buf = self._buf("send", self.world * cap, xp)
        torch.index_select(xp, 0, src, out=send_buf)
        return Routed(T, r.ids, r.weights, r.counts, r.offsets, r.perm, r.slot, counts, send_buf)

    def compute(self, recv_rows, recv_counts: torch.Tensor):
        """Expert FFN of the rows received from every source ([G, El] counts
        on the device).  exact: recv_rows holds the rows back to back, the
        outputs come back in the same order.  padded: block s of recv_rows
        holds source s's rows, and block s of the result its outputs."""
        seg = segment_offsets(recv_counts)
        n_seg = recv_counts.numel()
        if not self.padded:
            return self.ops.expert_ffn(recv_rows, seg, n_seg)
        cap = recv_rows.shape[0] // self.world
        n_s = recv_counts.sum(dim=1).long()                 # rows from each source
        pre = torch.zeros(self.world + 1, dtype=torch.long, device=n_s.device)
        torch.cumsum(n_s, 0, out=pre[1:])
        # pack the received blocks back to back: packed[q] = block s, row q - pre[s]
        q = self._ramp(self.world * cap, recv_rows.device)
        s = torch.searchsorted(pre[1:], q, right=True).clamp_(max=self.world - 1)
        src = torch.where(q < pre[-1], s * cap + (q - pre[s]), torch.zeros_like(q))
        packed = self._buf("packed", self.world * cap, recv_rows)
        torch.index_select(recv_rows, 0, src, out=packed)
        Y = self.ops.expert_ffn(packed, seg, n_seg)
        # and unpack: block s of the result = source s's outputs, in its order
        d = q // cap
        j = q - d * cap
        src2 = torch.where(j < n_s[d], pre[d] + j, torch.zeros_like(j))
        back_send = self._buf("back_send", self.world * cap, Y)
        torch.index_select(Y, 0, src2, out=back_send)
        return back_send

    def finish(self, routed: Routed, Y_back):
        """Combine this rank's tokens from its expert outputs.  exact: Y_back
        is the kept rows in dispatch order; padded: block d holds the outputs
        of the rows sent to rank d."""
        T, k = routed.T, self.ops.k
        full = self._buf("Y_full", max(T * k, 1), Y_back)[: T * k]
        if not self.padded:
            full[: Y_back.shape[0]] = Y_back
            return self.ops.combine(full, routed, T)
        cap = Y_back.shape[0] // self.world
        start = routed.offsets[:-1].reshape(self.world, self.El)[:, 0].long()
        rr = self._ramp(max(T * k, 1), Y_back.device)[: T * k]
        # dispatch row rr belongs to the destination whose slice holds it
        d = (torch.searchsorted(start, rr, right=True) - 1).clamp_(min=0)
        src = torch.where(rr < routed.offsets[-1].long(), d * cap + (rr - start[d]),
                          torch.zeros_like(rr))
        torch.index_select(Y_back, 0, src, out=full)
        return self.ops.combine(full, routed, T)

    # -- the whole layer -------------------------------------------------------

    def forward(self, x):
        routed = self.send(x)
        recv_counts = self.exchange.counts(routed.send_counts)
        if self.padded:
            recv = self.exchange.rows_even(routed.rows, self._buf("recv", routed.rows.shape[0],
                                                                  routed.rows))
            back_send = self.compute(recv, recv_counts)
            back = self.exchange.rows_even(back_send, self._buf("back", back_send.shape[0],
                                                                back_send))
            return self.finish(routed, back)
        # the step's one host read: the row splits of both directions
        splits = torch.stack([routed.send_counts.sum(dim=1), recv_counts.sum(dim=1)]).cpu()
        send_split, recv_split = splits[0].tolist(), splits[1].tolist()
        kept = sum(send_split)
        recv_rows = self.exchange.rows(routed.rows[:kept], send_split, recv_split)
        Y = self.compute(recv_rows, recv_counts)
        Y_back = self.exchange.rows(Y, recv_split, send_split)
        return self.finish(routed, Y_back)
