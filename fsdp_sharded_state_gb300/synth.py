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
              bf16 parameters and gradients, fp32 state; the fp32-parameter variant
              (suffix _p32: fp32 parameters = master, bf16 gradients; _p32g32: fp32
              gradients too).
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


SWEEP_DTYPES = {"": (torch.bfloat16, torch.bfloat16), "_p32": (torch.float32, torch.bfloat16),
                "_p32g32": (torch.float32, torch.float32)}


def sweep(P: int, N: int, param_dtype=torch.bfloat16, grad_dtype=torch.bfloat16) -> Workload:
    """One flat unit of P elements.  Default: bf16 parameters (fp32 master) and bf16
    gradients; param_dtype float32 is the fp32-parameter variant (the master is the
    parameter), with bf16 gradients as the workload states or fp32 ones."""
    suffix = {v: k for k, v in SWEEP_DTYPES.items()}[(param_dtype, grad_dtype)]
    return Workload(f"sweep_P{P}_N{N}{suffix}", 5, [(P,)], [0], N, FLAT, param_dtype, grad_dtype, 1, 1e-3)


def dim0_n6_h2048() -> Workload:
    """The dim-0 group at hidden 2048 (ffn 5504, vocab 32000; 93.6M parameters): the same
    dtypes, N and placement rule on a layout small enough for a profiler capture."""
    w = dim0_n6(hidden=2048, ffn=5504)
    w.name = "dim0_n6_h2048"
    return w


WORKLOADS = {"tiny_mlp": tiny_mlp, "mlp128m": mlp128m, "llama4": llama4, "dim0_n6": dim0_n6,
             "dim0_n6_h2048": dim0_n6_h2048}


def workload(name: str) -> Workload:
    """A workload by name; sweep points are named sweep_P<numel>_N<ranks>."""
    if name in WORKLOADS:
        return WORKLOADS[name]()
    if name.startswith("sweep_P"):
        p, rest = name[len("sweep_P"):].split("_N")
        n, suffix = (rest.split("_", 1) + [""])[:2]
        return sweep(int(p), int(n), *SWEEP_DTYPES["_" + suffix if suffix else ""])
    raise KeyError(f"unknown workload {name!r}: {sorted(WORKLOADS)} or sweep_P<numel>_N<ranks>[_p32|_p32g32]")


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


# ---------------------------------------------------------------------------
# Crafted bit patterns for the edge cases of the fp32 arithmetic and the bf16 cast.
# Inputs only: the patterns are chosen, never computed from the method.
# ---------------------------------------------------------------------------
def _pattern(values):
    """The fp32 bit patterns of the given values."""
    import numpy as np
    return np.asarray(values, dtype=np.float32).view(np.uint32)


def special_params(n: int, seed: int):
    """n fp32 parameters (numpy): a quarter ordinary N(0, 0.02) values, the rest
    special bit patterns in a seeded mix -- exact bf16 round-to-nearest-even ties
    (low half 0x8000, both parities of the high half), their neighbours (0x7fff,
    0x8001), subnormals, +-0, +-Inf, quiet and signalling NaNs, the largest finite
    values (which round up to Inf in bf16), the smallest normals, and large finite
    magnitudes (1e19 .. 3e38)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(n) * 0.02).astype(np.float32)
    kind = rng.integers(0, 12, n)
    sign = rng.integers(0, 2, n).astype(np.uint32) << 31
    hi = rng.integers(0x0080, 0x7F7F, n).astype(np.uint32)          # a normal bf16 high half
    u = x.view(np.uint32).copy()
    pick = {
        1: (hi << 16) | 0x8000,                                      # tie
        2: (hi << 16) | 0x7FFF,                                      # just below a tie
        3: (hi << 16) | 0x8001,                                      # just above a tie
        4: sign | rng.integers(1, 1 << 23, n).astype(np.uint32),    # subnormal
        5: sign,                                                     # +-0
        6: sign | 0x7F800000,                                        # +-Inf
        7: sign | 0x7FC00000 | rng.integers(0, 1 << 22, n).astype(np.uint32),   # quiet NaN
        8: sign | 0x7F800000 | rng.integers(1, 1 << 22, n).astype(np.uint32),   # signalling NaN
        9: sign | np.where(rng.integers(0, 2, n) == 1, 0x7F7FFFFF, 0x7F7F8000).astype(np.uint32),   # max finite, max tie
        10: sign | 0x00800000 | rng.integers(0, 2, n).astype(np.uint32) << 16,  # smallest normals
        11: sign | rng.choice(_pattern([1e19, 1e20, 1e21, 1e30, 3e38]), n),
    }
    for k, v in pick.items():
        sel = kind == k
        u[sel] = np.asarray(v, np.uint32)[sel]
    return u.view(np.float32)


def special_grads(n: int, N: int, seed: int, dtype: str = "f32"):
    """N gradient replicas of n elements (numpy; fp32, or bf16 as uint16 high halves)
    with, position by position, one seeded scenario: ordinary N(0, 1e-3) values; all
    replicas +-0; all replicas subnormal; one replica +Inf or -Inf; one replica +Inf
    and another -Inf; one replica NaN; all replicas near the fp32 maximum (their sum
    overflows); all replicas of magnitude 1e19 .. 1e21 (the squared term overflows);
    magnitudes 1e-20 .. 1e-30 (the squared term underflows)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    g = (rng.standard_normal((N, n)) * 1e-3).astype(np.float32)
    u = g.view(np.uint32)
    scen = rng.integers(0, 10, n)
    sign = lambda: rng.integers(0, 2, (N, n)).astype(np.uint32) << 31
    q1 = rng.integers(0, N, n)
    q2 = (q1 + 1 + rng.integers(0, max(N - 1, 1), n)) % N if N > 1 else q1
    cols = np.arange(n)
    if dtype == "bf16":
        sub = rng.integers(1, 1 << 7, (N, n)).astype(np.uint32) << 16      # bf16 subnormals
    else:
        sub = rng.integers(1, 1 << 23, (N, n)).astype(np.uint32)
    s = scen == 1
    u[:, s] = sign()[:, s]
    s = scen == 2
    u[:, s] = (sign() | sub)[:, s]
    s = scen == 3
    u[q1[s], cols[s]] = 0x7F800000 | (rng.integers(0, 2, s.sum()).astype(np.uint32) << 31)
    s = (scen == 4) & (q1 != q2)
    u[q1[s], cols[s]] = 0x7F800000
    u[q2[s], cols[s]] = 0xFF800000
    s = scen == 5
    u[q1[s], cols[s]] = 0x7FC00000 | rng.integers(0, 1 << 16, s.sum()).astype(np.uint32) << 6
    s = scen == 6
    big = np.uint32(0x7F7F0000) | (rng.integers(0, 1 << 16, (N, n)).astype(np.uint32) if dtype != "bf16" else 0)
    u[:, s] = (sign() | big)[:, s]
    s = scen == 7
    u[:, s] = (sign() | rng.choice(_pattern([1e19, 5e19, 1e20, 1e21]), (N, n)))[:, s]
    s = scen == 8
    u[:, s] = (sign() | rng.choice(_pattern([1e-20, 1e-25, 1e-30]), (N, n)))[:, s]
    if dtype == "bf16":
        # keep the high halves; a value whose low half is not zero rounds in the test's
        # own conversion, so clear it here: every pattern above is then a bf16 value
        return [(u[q] >> 16).astype(np.uint16) for q in range(N)]
    return [u[q].view(np.float32).copy() for q in range(N)]
