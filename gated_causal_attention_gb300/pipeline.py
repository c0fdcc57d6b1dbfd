"""Streaming batches from host memory through one entry point of the library and back.

For callers whose inputs start on the host and whose results must end there. Each step
uploads its inputs from pinned host memory, runs the call, and reads its outputs back to
pinned host memory. Three CUDA streams (uploads, compute, downloads) and `depth` sets of
device buffers let step k's call run while step k+1 uploads and step k-1 downloads; every
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
    complete once synchronize() returns (or the step's download event has completed)."""

    def __init__(self, call: Callable, in_specs: List[Spec], out_specs: List[Spec],
                 device=None, depth: int = 2):
        if depth < 1:
            raise ValueError("depth must be at least 1")
        self.device = torch.device(device if device is not None else "cuda")
        self.call = call
        self.depth = depth
        self.dev_in = [[torch.empty(tuple(s), dtype=dt, device=self.device) for s, dt in in_specs]
                       for _ in range(depth)]
        self.dev_out = [[torch.empty(tuple(s), dtype=dt, device=self.device) for s, dt in out_specs]
                        for _ in range(depth)]
        self.up = torch.cuda.Stream(self.device)
        self.comp = torch.cuda.Stream(self.device)
        self.down = torch.cuda.Stream(self.device)
        self.ev_up = [torch.cuda.Event() for _ in range(depth)]
        self.ev_comp = [torch.cuda.Event() for _ in range(depth)]
        self.ev_down = [torch.cuda.Event() for _ in range(depth)]
        self.steps = 0
        # the buffers were made on the current stream: the three streams start after that
        cur = torch.cuda.current_stream(self.device)
        for s in (self.up, self.comp, self.down):
            s.wait_stream(cur)

    def submit(self, host_inputs: Sequence[torch.Tensor], host_outputs: Sequence[torch.Tensor]):
        k, s = self.steps, self.steps % self.depth
        if k >= self.depth:
            self.up.wait_event(self.ev_comp[s])    # step k - depth has read these inputs
        with torch.cuda.stream(self.up):
            for d, h in zip(self.dev_in[s], host_inputs):
                d.copy_(h, non_blocking=True)
            self.ev_up[s].record(self.up)
        self.comp.wait_event(self.ev_up[s])
        if k >= self.depth:
            self.comp.wait_event(self.ev_down[s])  # step k - depth's outputs have left
        self.call(self.dev_in[s], self.dev_out[s], self.comp)
        self.ev_comp[s].record(self.comp)
        self.down.wait_event(self.ev_comp[s])
        with torch.cuda.stream(self.down):
            for h, d in zip(host_outputs, self.dev_out[s]):
                h.copy_(d, non_blocking=True)
            self.ev_down[s].record(self.down)
        self.steps += 1
        return self.ev_down[s]

    def synchronize(self):
        for s in (self.up, self.comp, self.down):
            s.synchronize()
