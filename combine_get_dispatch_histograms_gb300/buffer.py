"""The event-driven call protocol of the pages' Buffer, over Context.

Page "DeepEP 学习笔记", section "三个方法概览": every method switches to a
communication stream after the previous event, launches its work there, and
either returns an event handle (asynchronous) or makes the compute stream
wait for it; dispatch waits on the host for the receive counts between the
notify and the copy and returns the handle that combine uses.  Buffer gives
that protocol to Context's calls; the work itself is the library's kernels.
Tensors that the communication stream uses are recorded on it, so the
caching allocator does not reuse them before that stream is done.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import Context


class EventOverlap:
    """A CUDA event recorded after a call's work on the communication stream."""

    def __init__(self, event: Optional[torch.cuda.Event]):
        self.event = event

    def current_stream_wait(self) -> None:
        """Make the current (compute) stream wait for the call's work."""
        if self.event is not None:
            torch.cuda.current_stream().wait_event(self.event)


@dataclass
class DispatchResult:
    recv: dict            # recv_x and its metadata (the receive layout)
    handle: object        # the notify handle (combine routes back with it)
    layout: dict          # the layout histograms
    event: EventOverlap


class Buffer:
    """get_dispatch_layout / dispatch / combine on a communication stream."""

    def __init__(self, ctx: Context, comm_stream: Optional[torch.cuda.Stream] = None):
        self.ctx = ctx
        self.comm = comm_stream if comm_stream is not None else torch.cuda.Stream(device=ctx.device)

    def _enter(self, previous_event: Optional[EventOverlap]):
        compute = torch.cuda.current_stream()
        if previous_event is not None and previous_event.event is not None:
            self.comm.wait_event(previous_event.event)
        else:
            self.comm.wait_stream(compute)
        return compute

    def _leave(self, compute, async_finish: bool, tensors) -> EventOverlap:
        ev = torch.cuda.Event()
        ev.record(self.comm)
        for t in tensors:
            if isinstance(t, torch.Tensor) and t.is_cuda:
                t.record_stream(self.comm)
        if not async_finish:
            compute.wait_event(ev)
        return EventOverlap(ev)

    def get_dispatch_layout(self, topk_idx: torch.Tensor, previous_event: Optional[EventOverlap] = None,
                            async_finish: bool = False):
        """Returns (layout dict, event)."""
        compute = self._enter(previous_event)
        with torch.cuda.stream(self.comm):
            lay = self.ctx.get_dispatch_layout(topk_idx)
        return lay, self._leave(compute, async_finish, [topk_idx, *lay.values()])

    def dispatch(self, x: torch.Tensor, topk_idx: torch.Tensor, topk_weights: torch.Tensor,
                 layout: Optional[dict] = None, previous_event: Optional[EventOverlap] = None,
                 async_finish: bool = False) -> DispatchResult:
        """Notify (waiting on the host for the receive counts), then the scatter
        (the staged one with nodes)."""
        compute = self._enter(previous_event)
        with torch.cuda.stream(self.comm):
            if layout is None:
                layout = self.ctx.get_dispatch_layout(topk_idx)
            h = self.ctx.notify_dispatch(topk_idx, layout)
            if self.ctx.N > 1:  # hierarchical: node staging, then the ranks of the node
                recv = self.ctx.dispatch_hier(x, topk_idx, topk_weights, h)
            else:
                recv = self.ctx.dispatch(x, topk_idx, topk_weights, h)
        ev = self._leave(compute, async_finish,
                         [x, topk_idx, topk_weights, *layout.values(), *h.values(), *recv.values()])
        return DispatchResult(recv, h, layout, ev)

    def permute(self, result: DispatchResult, previous_event: Optional[EventOverlap] = None,
                async_finish: bool = False):
        """Received rows into per-expert blocks; returns (permuted dict, event)."""
        compute = self._enter(previous_event)
        with torch.cuda.stream(self.comm):
            perm = self.ctx.permute(result.handle, result.recv)
        return perm, self._leave(compute, async_finish, [*result.recv.values(), *perm.values()])

    def combine(self, result: DispatchResult, expert_out: torch.Tensor, topk_idx: torch.Tensor,
                topk_weights: torch.Tensor, previous_event: Optional[EventOverlap] = None,
                async_finish: bool = False):
        """The weighted reduction back to token order; returns (out, event)."""
        compute = self._enter(previous_event)
        with torch.cuda.stream(self.comm):
            out = self.ctx.combine(result.handle, expert_out, topk_idx, topk_weights, hier=self.ctx.N > 1)
        return out, self._leave(compute, async_finish, [expert_out, topk_idx, topk_weights, out])
