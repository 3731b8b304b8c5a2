"""Running the layer over a sequence of token batches that live in host
memory, with the host<->device copies overlapped with the computation.

While batch i is computed, batch i+1's tokens travel to the device and
batch i-1's output travels back: two device slots for x and y, one stream
per direction of copy, and events that keep each slot's uses in order.  The
kernels are the layer's own (moe_forward); this only schedules the copies
around them, as a serving loop would.
"""
from __future__ import annotations

import torch

from . import moe_forward


class HostPipeline:
    """Moves host batches of T tokens through `layer` (a MoELayer on
    `device`), two batches in flight."""

    SLOTS = 2

    def __init__(self, layer, T: int, device, graphs: bool = False):
        """graphs: replay, per device slot, a CUDA graph of the slot's forward
        (captured here, after one eager call) instead of launching its
        kernels from the host each batch."""
        self.layer = layer
        self.device = torch.device(device)
        layer._ensure(T, self.device)
        self.T = T
        bf = dict(dtype=torch.bfloat16, device=self.device)
        self.x_dev = [torch.zeros(T, layer.H, **bf) for _ in range(self.SLOTS)]
        self.y_dev = [torch.empty(T, layer.H, **bf) for _ in range(self.SLOTS)]
        self.h2d = torch.cuda.Stream(self.device)
        self.d2h = torch.cuda.Stream(self.device)
        self.graphs = None
        if graphs:
            cap = torch.cuda.Stream(self.device)
            cap.wait_stream(torch.cuda.current_stream(self.device))
            self.graphs = []
            for s in range(self.SLOTS):
                self._forward(s, cap)  # eager first: one-time library setup stays out of capture
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap):
                    self._forward(s, cap)
                self.graphs.append(g)
            torch.cuda.current_stream(self.device).wait_stream(cap)

    def _forward(self, s: int, stream):
        L, r = self.layer, self.layer.routing
        moe_forward(L.shape, self.x_dev[s], L.w_router, L.bias, L.w1, L.w2, self.y_dev[s],
                    r.ids, r.weights, r.counts, r.offsets, r.perm, r.slot, L.ws, stream)

    def run(self, x_hosts, y_hosts, stream=None):
        """y_hosts[i] <- layer(x_hosts[i]) for every i; host tensors pinned,
        [T, H] bf16.  Enqueues everything and returns without waiting;
        synchronise `stream` (default: the current stream) to wait for the
        last output."""
        cs = stream or torch.cuda.current_stream(self.device)
        up = [torch.cuda.Event() for _ in range(self.SLOTS)]      # x slot filled
        done = [torch.cuda.Event() for _ in range(self.SLOTS)]    # slot computed
        down = [torch.cuda.Event() for _ in range(self.SLOTS)]    # y slot read back
        for e in done + down:
            e.record(cs)
        for i, (xh, yh) in enumerate(zip(x_hosts, y_hosts)):
            s = i % self.SLOTS
            self.h2d.wait_event(done[s])  # the slot's previous batch has been computed
            with torch.cuda.stream(self.h2d):
                self.x_dev[s].copy_(xh, non_blocking=True)
            up[s].record(self.h2d)
            cs.wait_event(up[s])
            cs.wait_event(down[s])  # its previous output has been read back
            if self.graphs is None:
                self._forward(s, cs)
            else:
                with torch.cuda.stream(cs):
                    self.graphs[s].replay()
            done[s].record(cs)
            self.d2h.wait_event(done[s])
            with torch.cuda.stream(self.d2h):
                yh.copy_(self.y_dev[s], non_blocking=True)
            down[s].record(self.d2h)
        for e in down:
            cs.wait_event(e)
