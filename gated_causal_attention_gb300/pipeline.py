"""Streaming batches from host memory through one entry point of the library and back.

For callers whose inputs start on the host and whose results must end there. Each step
uploads its inputs from pinned host memory, runs the call, and reads its outputs back to
pinned host memory. Upload streams, a compute stream and download streams with `depth` sets
of device buffers let step k's call run while step k+1 uploads and step k-1 downloads; every
step still moves all of its bytes, and each call sees exactly the inputs of its own step, so
the results are those of running the steps one after another.

This is plumbing (device buffers, streams, events); the computation is the call's.
"""
from __future__ import annotations

from typing import Callable, List, Sequence, Tuple

import torch

Spec = Tuple[Sequence[int], torch.dtype]


class HostPipeline:
    """call(dev_inputs, dev_outputs, stream) enqueues one step's work on `stream`, reading the
    device tensors dev_inputs and writing dev_outputs (shapes and dtypes from in_specs and
    out_specs). submit(host_inputs, host_outputs) queues one step; host tensors should be
    pinned (page-locked) so that the copies are asynchronous, and a step's host outputs are
    complete once synchronize() returns (or the event submit() returns has completed).

    Each direction spreads its tensors over `copy_streams` streams (tensor i on stream
    i % copy_streams, tensors of 8 MiB and more cut into that many pieces), so that several copy engines
    move one step's bytes at once."""

    def __init__(self, call: Callable, in_specs: List[Spec], out_specs: List[Spec],
                 device=None, depth: int = 2, copy_streams: int = 1):
        if depth < 1 or copy_streams < 1:
            raise ValueError("depth and copy_streams must be at least 1")
        self.device = torch.device(device if device is not None else "cuda")
        self.call = call
        self.depth = depth
        self.nc = copy_streams
        self.dev_in = [[torch.empty(tuple(s), dtype=dt, device=self.device) for s, dt in in_specs]
                       for _ in range(depth)]
        self.dev_out = [[torch.empty(tuple(s), dtype=dt, device=self.device) for s, dt in out_specs]
                        for _ in range(depth)]
        self.up = [torch.cuda.Stream(self.device) for _ in range(self.nc)]
        self.comp = torch.cuda.Stream(self.device)
        self.down = [torch.cuda.Stream(self.device) for _ in range(self.nc)]
        self.ev_up = [[torch.cuda.Event() for _ in range(self.nc)] for _ in range(depth)]
        self.ev_comp = [torch.cuda.Event() for _ in range(depth)]
        self.ev_down = [[torch.cuda.Event() for _ in range(self.nc)] for _ in range(depth)]
        self.steps = 0
        # the buffers were made on the current stream: every stream starts after that
        cur = torch.cuda.current_stream(self.device)
        for s in self.up + self.down + [self.comp]:
            s.wait_stream(cur)

    def _pieces(self, dst, src):
        """(dst, src) cut into up to copy_streams equal pieces of their flattened elements
        (both contiguous); tensors under 8 MiB stay whole."""
        n = dst.numel()
        if self.nc == 1 or n * dst.element_size() < (8 << 20):
            return [(dst, src)]
        d, h = dst.view(-1), src.view(-1)
        cuts = [n * i // self.nc for i in range(self.nc + 1)]
        return [(d[a:b], h[a:b]) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]

    def _copies(self, pairs, streams):
        jobs = []
        for d, h in pairs:
            jobs.extend(self._pieces(d, h))
        for i, (d, h) in enumerate(jobs):
            with torch.cuda.stream(streams[i % self.nc]):
                d.copy_(h, non_blocking=True)

    def submit(self, host_inputs: Sequence[torch.Tensor], host_outputs: Sequence[torch.Tensor]):
        k, s = self.steps, self.steps % self.depth
        for c, st in enumerate(self.up):
            if k >= self.depth:
                st.wait_event(self.ev_comp[s])    # step k - depth has read these inputs
        self._copies(list(zip(self.dev_in[s], host_inputs)), self.up)
        for c, st in enumerate(self.up):
            self.ev_up[s][c].record(st)
            self.comp.wait_event(self.ev_up[s][c])
        if k >= self.depth:
            for c in range(self.nc):
                self.comp.wait_event(self.ev_down[s][c])  # step k - depth's outputs have left
        self.call(self.dev_in[s], self.dev_out[s], self.comp)
        self.ev_comp[s].record(self.comp)
        for st in self.down:
            st.wait_event(self.ev_comp[s])
        self._copies(list(zip(host_outputs, self.dev_out[s])), self.down)
        for c, st in enumerate(self.down):
            self.ev_down[s][c].record(st)
        self.steps += 1
        return self.ev_down[s]

    def synchronize(self):
        for s in self.up + self.down + [self.comp]:
            s.synchronize()
