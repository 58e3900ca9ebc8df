"""HostFeed: sharded steps on gradients that arrive in host memory.

A training loop whose gradient replicas are produced on the host (or staged
there) pays for the host link every step: the N replicas go host -> device, and
each step's result (the updated parameter shards) comes back.  On GB300 each
direction of the link streams at about 0.2 TB/s; one H2D stream alone gets well
under that, two or more reach it.  HostFeed overlaps the link with the step:

  * the replicas of step k go into device buffer k mod 2 on two H2D streams,
    while step k-1 computes and its parameters go back on a D2H stream;
  * step k's reduce-scatter waits until the D2H of step k-1 has read the
    parameter shards it overwrites, and buffer k mod 2 is refilled only once
    step k's reduce-scatter has read it.

It is plumbing over ShardedState (torch streams and events); every step runs
the library's unshard and fused reduce-scatter + AdamW + cast kernels.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from .state import STRATEGIES, ShardedState


class HostFeed:
    def __init__(self, state: ShardedState, grad_dtype: torch.dtype, n_buffers: int = 2, copy_streams: int = 2,
                 stream: Optional[torch.cuda.Stream] = None):
        if n_buffers < 1 or copy_streams < 1:
            raise ValueError("n_buffers and copy_streams must be >= 1")
        self.st = state
        dev = state.full.device
        self.bufs = [[torch.empty(state.F, dtype=grad_dtype, device=dev) for _ in range(state.N)]
                     for _ in range(n_buffers)]
        self.h2d = [torch.cuda.Stream(dev) for _ in range(copy_streams)]
        self.d2h = torch.cuda.Stream(dev)
        self.compute = stream if stream is not None else torch.cuda.current_stream(dev)
        self.free = [None] * n_buffers        # buffer b may be refilled once this event has passed
        self.shards_read = None               # the previous step's D2H has read the parameter shards
        self.start = None
        self.k = 0

    def begin(self) -> None:
        """Orders the copies of the next steps after the work already on the compute stream."""
        self.start = torch.cuda.Event()
        self.start.record(self.compute)

    def step(self, host_grads: Sequence[torch.Tensor], out_host: torch.Tensor, hp, strategy: str = "full_shard",
             step: Optional[int] = None) -> None:
        """One step: H2D of the N pinned host replicas, the step's all-gathers, the
        fused reduce-scatter + AdamW + cast, and D2H of the updated parameter
        shards into the pinned out_host (the shape of state.param_shards)."""
        st = self.st
        if len(host_grads) != st.N:
            raise ValueError(f"need {st.N} gradient replicas, got {len(host_grads)}")
        if self.start is None:
            self.begin()
        b = self.k % len(self.bufs)
        bufs = self.bufs[b]
        ready = []
        for i, s in enumerate(self.h2d):
            s.wait_event(self.free[b] if self.free[b] is not None else self.start)
            with torch.cuda.stream(s):
                for q in range(i, st.N, len(self.h2d)):
                    bufs[q].copy_(host_grads[q], non_blocking=True)
            e = torch.cuda.Event()
            e.record(s)
            ready.append(e)
        cs = self.compute
        for e in ready:
            cs.wait_event(e)
        for _ in range(STRATEGIES[strategy]):
            st.unshard(stream=cs)
        if self.shards_read is not None:
            cs.wait_event(self.shards_read)
        st.reduce_scatter_adamw(bufs, hp, step=step, stream=cs)
        done = torch.cuda.Event()
        done.record(cs)
        self.free[b] = done
        self.d2h.wait_event(done)
        with torch.cuda.stream(self.d2h):
            out_host.copy_(st.param_shards, non_blocking=True)
        self.shards_read = torch.cuda.Event()
        self.shards_read.record(self.d2h)
        self.k += 1

    def finish(self) -> None:
        """Makes the compute stream wait for every copy issued so far."""
        for s in self.h2d:
            self.compute.wait_stream(s)
        self.compute.wait_stream(self.d2h)
        self.start = None
