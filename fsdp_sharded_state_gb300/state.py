"""ShardedState: the buffers of one sharded model state and the step that uses them.

Harness over the C-ABI calls: it allocates the [N][stride] shard arrays and the
full buffer with torch (device memory is all torch is used for) and issues the
library calls of one training step in the order the FSDP pages give
("第18章 FSDP：ZeRO 风格的参数分片" §18.2/§18.3/§18.21; "NCCL ZeRO/FSDP state
sharding", sections "ZeRO-2 方向" and "ZeRO-3 方向"):

    FULL_SHARD     unshard (forward) -> unshard (backward) -> reduce-scatter+AdamW+cast
    SHARD_GRAD_OP  unshard (forward)                      -> reduce-scatter+AdamW+cast

The gradients are the caller's: in a model they come out of backward; here they
are given as N full-layout replicas, one per simulated rank.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import (FSDP_BF16, FSDP_F32, FSDP_FLAT, Layout, fsdp_adamw_step_consts_make, fsdp_reduce_scatter_adamw,
               fsdp_reduce_scatter_adamw_consts, fsdp_reshard, fsdp_rs_kernel_for, fsdp_unshard)

STRATEGIES = {"full_shard": 2, "shard_grad_op": 1}   # all-gathers per step


def step_schedule(n_units: int, strategy: str = "full_shard"):
    """The per-unit collectives of one step, in the order FSDP issues them, as
    ("all_gather", u) / ("reduce_scatter", u) pairs.  Forward gathers every unit in
    order; backward visits the units in reverse, and under FULL_SHARD gathers each
    one again first (the forward freed it), then reduce-scatters its gradient;
    SHARD_GRAD_OP keeps the forward gather through backward ("NCCL ZeRO/FSDP state
    sharding", sections "ZeRO-2 方向" and "ZeRO-3 方向": with 8 wrap units, 8 + 0
    all-gathers and 8 reduce-scatters, and 8 + 8 all-gathers and 8 reduce-scatters)."""
    if strategy not in STRATEGIES:
        raise ValueError(f"unknown strategy {strategy!r}")
    sched = [("all_gather", u) for u in range(n_units)]
    for u in reversed(range(n_units)):
        if strategy == "full_shard":
            sched.append(("all_gather", u))
        sched.append(("reduce_scatter", u))
    return sched


class ShardedState:
    def __init__(self, shapes: Sequence[Sequence[int]], unit_ids: Optional[Sequence[int]], n_ranks: int,
                 mode: int = FSDP_FLAT, param_dtype: torch.dtype = torch.bfloat16, device="cuda",
                 with_grad_out: bool = False):
        if param_dtype not in (torch.bfloat16, torch.float32):
            raise TypeError("param_dtype must be bfloat16 or float32")
        code = FSDP_BF16 if param_dtype == torch.bfloat16 else FSDP_F32
        self.layout = Layout(shapes, unit_ids, n_ranks, mode, [code] * len(shapes))
        self.N, self.stride = n_ranks, self.layout.stride
        self.F = self.layout.info["full_numel"]
        self.P = self.layout.info["numel"]
        self.param_dtype = param_dtype
        dev = torch.device(device)
        z = lambda dt: torch.zeros(self.N, self.stride, dtype=dt, device=dev)
        self.master, self.exp_avg, self.exp_avg_sq = z(torch.float32), z(torch.float32), z(torch.float32)
        self.param = z(torch.bfloat16) if param_dtype == torch.bfloat16 else None
        self.grad_out = z(torch.float32) if with_grad_out else None
        self.full = torch.zeros(self.F, dtype=param_dtype, device=dev)
        self.t = 0

    @property
    def param_shards(self) -> torch.Tensor:
        """What the all-gather reads: the bf16 copies, or the fp32 master itself."""
        return self.param if self.param is not None else self.master

    def units(self, ub: int = 0, ue: Optional[int] = None):
        return ub, self.layout.n_units if ue is None else ue

    def init_from_full(self, full: torch.Tensor, stream=None) -> None:
        """Initial sharding of a constructed model (fp32 or bf16 full layout); moments to zero."""
        fsdp_reshard(self.layout, 0, self.layout.n_units, full, self.master, self.param, stream)
        self.exp_avg.zero_()
        self.exp_avg_sq.zero_()
        self.t = 0

    def unshard(self, ub: int = 0, ue: Optional[int] = None, out: Optional[torch.Tensor] = None, stream=None):
        ub, ue = self.units(ub, ue)
        fsdp_unshard(self.layout, ub, ue, self.param_shards, self.full if out is None else out, stream)
        return self.full if out is None else out

    def reduce_scatter_adamw(self, grads, hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step: Optional[int] = None,
                             ub: int = 0, ue: Optional[int] = None, stream=None) -> None:
        ub, ue = self.units(ub, ue)
        t = self.t + 1 if step is None else step
        fsdp_reduce_scatter_adamw(self.layout, ub, ue, grads, self.master, self.exp_avg, self.exp_avg_sq,
                                  self.param, self.grad_out, hp, t, stream)
        self.t = t

    def step(self, grads, hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), strategy: str = "full_shard", stream=None) -> None:
        """One sharded step over all units: the all-gathers of the strategy, then
        the fused reduce-scatter + AdamW + cast."""
        for _ in range(STRATEGIES[strategy]):
            self.unshard(stream=stream)
        self.reduce_scatter_adamw(grads, hp, stream=stream)

    def step_per_unit(self, grads, hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), strategy: str = "full_shard",
                      stream=None, gather_stream=None) -> None:
        """The same step issued unit by unit, in step_schedule's order: one library call
        per collective of the pages' per-unit FSDP schedule, every reduce-scatter with
        the same step number.  Same results as step(), bit for bit.

        With gather_stream, the all-gathers go on that stream and the reduce-scatters on
        `stream` (the current one by default), as FSDP keeps its all-gathers on a
        stream of their own ([FSDP-ch18] §18.3, prefetch): a unit's reduce-scatter
        waits for that unit's last all-gather (it rewrites the shards the gather reads),
        and the step's gathers wait for all work queued on `stream` before the step (the
        previous step's updates).  So the gather of unit u-1 runs beside the
        reduce-scatter of unit u.  When the call returns, `stream` holds the whole step."""
        t = self.t + 1
        if gather_stream is None:
            for kind, u in step_schedule(self.layout.n_units, strategy):
                if kind == "all_gather":
                    self.unshard(u, u + 1, stream=stream)
                else:
                    self.reduce_scatter_adamw(grads, hp, step=t, ub=u, ue=u + 1, stream=stream)
            self.t = t
            return
        main = stream if stream is not None else torch.cuda.current_stream(self.full.device)
        gather_stream.wait_stream(main)
        gathered = {}
        for kind, u in step_schedule(self.layout.n_units, strategy):
            if kind == "all_gather":
                self.unshard(u, u + 1, stream=gather_stream)
                ev = torch.cuda.Event()
                ev.record(gather_stream)
                gathered[u] = ev                  # the unit's latest gather
            else:
                main.wait_event(gathered[u])
                self.reduce_scatter_adamw(grads, hp, step=t, ub=u, ue=u + 1, stream=main)
        main.wait_stream(gather_stream)           # the step's last gathers, for the caller
        self.t = t

    def launch_counts(self, grad_dtype: torch.dtype = torch.bfloat16) -> dict:
        """Kernels one call launches.  The all-gather and the direct reduce-scatter
        kernels: one per alignment class present (shard and full-layout offsets
        congruent mod 8 or not) -- the layout files every rank's piece under one of
        the two; the staged reduce-scatter kernel: one for both.  Plus the zero-fill
        of the gradient shard's padding when a gradient shard is written."""
        L, N, stride = self.layout, self.N, self.stride
        data, gather = set(), set()
        for t in range(len(L.shapes)):
            for r in range(N):
                sg = L.segment(t, r)
                if sg["len"]:
                    data.add((sg["full_off"] - (r * stride + sg["shard_off"])) % 8 == 0)
        if L.mode == 0:                      # FLAT: the all-gather copies whole S_u slots
            for u in range(L.n_units):
                d = L.unit(u)
                if d["shard_numel"]:
                    for r in range(N):
                        gather.add((d["full_off"] + r * d["shard_numel"] - (r * stride + d["shard_off"])) % 8 == 0)
        else:
            gather = set(data)
        pad = 1 if (self.grad_out is not None and self.layout.info["pad_numel"] + N * (stride - self.layout.info[
            "shard_numel"]) > 0) else 0
        staged = fsdp_rs_kernel_for(self.layout, grad_dtype) == "staged"
        rs = (1 if data else 0) if staged else len(data)
        return {"unshard": len(gather), "reduce_scatter_adamw": rs + pad}

    def launches_per_step(self, strategy: str = "full_shard", grad_dtype: torch.dtype = torch.bfloat16) -> int:
        """Kernel launches of one step (for a launch count)."""
        c = self.launch_counts(grad_dtype)
        return STRATEGIES[strategy] * c["unshard"] + c["reduce_scatter_adamw"]


class StepGraph:
    """One sharded step captured in CUDA graphs and replayed step after step.

    For layouts small enough that issuing a step's library calls takes the host longer
    than the GPU takes to run them (the 4,192-parameter MLP: about 30 us of host work
    for a step the GPU runs in about 10 us), the step's kernels are captured once and
    each step is one graph launch.  The fused update reads its AdamW step constants
    from a 48-byte block in page-locked host memory (fsdp_reduce_scatter_adamw_consts),
    which step() fills with the step's constants (fsdp_adamw_step_consts_make) before
    the replay; the graph holds no copy.  n_blocks host blocks, each with its own
    graph, take turns, so the host rewrites a block only once the replay that read it
    has run: it runs at most n_blocks steps ahead.

    The first step() runs the same calls eagerly (it also sets up the library's
    per-kernel launch state, which must not happen during capture); the graphs are
    captured right after it.  Buffers are fixed at construction: the step reads
    `grads` every time, as a training loop that refills them in place would.  Call
    step() with one current stream throughout: replays on two streams would update the
    same state concurrently.  Same results as ShardedState.step, bit for bit."""

    def __init__(self, state: ShardedState, grads, hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), strategy: str = "full_shard",
                 n_blocks: int = 3):
        if strategy not in STRATEGIES:
            raise ValueError(f"unknown strategy {strategy!r}")
        if n_blocks < 1:
            raise ValueError("n_blocks must be >= 1")
        self.st, self.grads, self.hp, self.strategy = state, list(grads), hp, strategy
        self.host = [torch.zeros(12, dtype=torch.float32).pin_memory() for _ in range(n_blocks)]
        self.done = [None] * n_blocks
        self.graphs = None
        self.k = 0
        state.layout.prepare()

    def _calls(self, b: int) -> None:
        st = self.st
        for _ in range(STRATEGIES[self.strategy]):
            st.unshard()
        fsdp_reduce_scatter_adamw_consts(st.layout, 0, st.layout.n_units, self.grads, st.master, st.exp_avg,
                                         st.exp_avg_sq, st.param, st.grad_out, consts=self.host[b])

    def _capture(self) -> None:
        torch.cuda.synchronize(self.st.full.device)
        graphs = []
        for b in range(len(self.host)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                self._calls(b)
            graphs.append(g)
        self.graphs = graphs

    def step(self) -> None:
        """One step: the next step number's constants into a host block, then the graph
        that reads that block (on the current stream)."""
        b = self.k % len(self.host)
        if self.done[b] is not None:
            self.done[b].synchronize()           # the replay that last read block b has run
        t = self.st.t + 1
        c = fsdp_adamw_step_consts_make(self.st.layout, self.hp, t)
        ctypes.memmove(self.host[b].data_ptr(), ctypes.addressof(c), ctypes.sizeof(c))
        if self.graphs is None:
            self._calls(b)
            torch.cuda.current_stream().synchronize()
            self._capture()
        else:
            self.graphs[b].replay()
        ev = torch.cuda.Event()
        ev.record()
        self.done[b] = ev
        self.st.t = t
        self.k += 1
