"""Seeded synthetic inputs and the workload recipes they follow.

This module holds none of the sharded-state arithmetic: it draws random numbers
and fills buffers at offsets it is given.  Both the CUDA path (tests, bench) and
the oracle (tests) take their inputs from here, so the two sides see the same
bytes.

Workloads (shapes of the pages' examples; values are synthetic, no weights):
  tiny_mlp    MLP of [64,32],[64],[32,64],[32] (4,192 elements) in one FLAT unit,
              N=4, fp32 parameters and gradients, 3 steps.
  mlp128m     8 Linear weights [2048,2048] fp32 = 128 MiB, each its own FLAT unit
              (one wrap unit per Linear), N=4, fp32 gradients and moments, 10 steps
              -- the 4-GPU experiment of "NCCL ZeRO/FSDP state sharding".
  llama4      4 Llama-style blocks (q,k,v,o [4096,4096]; gate,up [11008,4096];
              down [4096,11008]; attn/ffn RMSNorm weights [4096]), one FLAT unit per
              block, N=8, bf16 parameters and gradients, fp32 master and moments.
  dim0_n6     FSDP2 per-tensor dim-0 sharding of [32000,4096], 4x[4096,4096],
              [11008,4096], [4096] in one group, N=6 (rows not divisible by N),
              bf16 parameters and gradients, fp32 state.
  sweep       one flat unit of P elements (powers of two and +1), N in {2..32},
              bf16 parameters and gradients, fp32 state.
Value recipe: parameters ~ N(0, 0.02) (standard deviation), RMSNorm weights 1.0;
per-rank gradients ~ N(0, sigma) with sigma 1e-2 (tiny_mlp) or 1e-3, drawn in
fp32 and rounded to the gradient dtype by torch (nearest even).
Seeds: parameters 1000*cfg; gradients 1000*cfg + 100*step + rank.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import torch

HP = (1e-3, 0.9, 0.999, 1e-8, 0.01)   # AdamW lr, beta1, beta2, eps, weight_decay

FLAT, DIM0 = 0, 1


@dataclass
class Workload:
    name: str
    cfg_id: int
    shapes: List[Tuple[int, ...]]
    unit_ids: List[int]
    N: int
    mode: int
    param_dtype: torch.dtype
    grad_dtype: torch.dtype
    steps: int
    grad_std: float
    param_std: float = 0.02
    ones: List[int] = field(default_factory=list)     # tensors initialised to 1.0 (RMSNorm weights)
    hp: Tuple[float, ...] = HP

    @property
    def numel(self) -> int:
        n = 0
        for s in self.shapes:
            k = 1
            for d in s:
                k *= d
            n += k
        return n


def llama_block_shapes(hidden=4096, ffn=11008):
    return [(hidden, hidden)] * 4 + [(ffn, hidden), (ffn, hidden), (hidden, ffn), (hidden,), (hidden,)]


def tiny_mlp(mode=FLAT) -> Workload:
    return Workload("tiny_mlp", 1, [(64, 32), (64,), (32, 64), (32,)], [0, 0, 0, 0], 4, mode,
                    torch.float32, torch.float32, 3, 1e-2)


def mlp128m() -> Workload:
    return Workload("mlp128m", 2, [(2048, 2048)] * 8, list(range(8)), 4, FLAT,
                    torch.float32, torch.float32, 10, 1e-3)


def llama4(blocks=4, hidden=4096, ffn=11008, N=8) -> Workload:
    shapes, units, ones = [], [], []
    for b in range(blocks):
        for s in llama_block_shapes(hidden, ffn):
            if len(s) == 1:
                ones.append(len(shapes))
            shapes.append(s)
            units.append(b)
    return Workload("llama4", 3, shapes, units, N, FLAT, torch.bfloat16, torch.bfloat16, 3, 1e-3, ones=ones)


def dim0_n6(vocab=32000, hidden=4096, ffn=11008, N=6) -> Workload:
    shapes = [(vocab, hidden)] + [(hidden, hidden)] * 4 + [(ffn, hidden), (hidden,)]
    return Workload("dim0_n6", 4, shapes, [0] * len(shapes), N, DIM0, torch.bfloat16, torch.bfloat16, 3, 1e-3)


def sweep(P: int, N: int) -> Workload:
    return Workload(f"sweep_P{P}_N{N}", 5, [(P,)], [0], N, FLAT, torch.bfloat16, torch.bfloat16, 1, 1e-3)


WORKLOADS = {"tiny_mlp": tiny_mlp, "mlp128m": mlp128m, "llama4": llama4, "dim0_n6": dim0_n6}


def workload(name: str) -> Workload:
    """A workload by name; sweep points are named sweep_P<numel>_N<ranks>."""
    if name in WORKLOADS:
        return WORKLOADS[name]()
    if name.startswith("sweep_P"):
        p, n = name[len("sweep_P"):].split("_N")
        return sweep(int(p), int(n))
    raise KeyError(f"unknown workload {name!r}: {sorted(WORKLOADS)} or sweep_P<numel>_N<ranks>")


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def full_params(w: Workload, full_numel: int, tensor_full_offsets: Sequence[int], device="cuda",
                dtype=torch.float32) -> torch.Tensor:
    """The full-layout parameter buffer: N(0, param_std) everywhere, then the
    tensors listed in w.ones set to 1.0 at the offsets given by the caller.
    Positions that hold no tensor (FLAT padding) keep random values: nothing may read them."""
    g = _gen(1000 * w.cfg_id, device)
    x = torch.randn(full_numel, generator=g, device=device, dtype=torch.float32) * w.param_std
    for t in w.ones:
        n = 1
        for d in w.shapes[t]:
            n *= d
        o = int(tensor_full_offsets[t])
        x[o:o + n] = 1.0
    return x.to(dtype)


def grad_replica(w: Workload, full_numel: int, step: int, rank: int, device="cuda",
                 out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Rank `rank`'s gradient at `step` (1-based) over the full layout, in w.grad_dtype.
    FLAT padding positions hold random values too: the reduce-scatter must not read them."""
    g = _gen(1000 * w.cfg_id + 100 * step + rank, device)
    x = torch.randn(full_numel, generator=g, device=device, dtype=torch.float32) * w.grad_std
    if out is None:
        return x.to(w.grad_dtype)
    out.copy_(x)
    return out


def grad_replicas(w: Workload, full_numel: int, step: int, device="cuda") -> List[torch.Tensor]:
    return [grad_replica(w, full_numel, step, r, device) for r in range(w.N)]
