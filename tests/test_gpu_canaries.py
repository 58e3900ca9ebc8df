"""Canary regions around every buffer every entry point writes (GPU).

Each output buffer sits inside a larger allocation whose margins (4 KB on each side)
hold a known bit pattern; after the calls the margins must be unchanged, so no kernel
wrote outside its buffer.  Covered: the reshard, the all-gather, the fused step (with
the reduced-gradient output), the sharded clip (the cooperative launch on an aligned
layout, the two passes on a misaligned one; its workspace and norm output too), the
accumulation, HSDP (R = 2) and ZeRO-1, under each kernel choice.  This is the library's
own out-of-bounds check for writes: the memory checker of the CUDA toolkit is not
available on this GPU pool.
"""
import pytest
import torch

import fsdp_sharded_state_gb300 as fs
from fsdp_sharded_state_gb300 import synth

import parity_util as pu

pytestmark = pytest.mark.gpu

PAD = 1024                      # elements of margin on each side
C32, C16, C8 = 0x5A5A5A5A, 0x5A5A, 0x5A


class Arenas:
    """Buffers carved from the middle of canary-filled allocations."""

    def __init__(self):
        self.all = {}

    def make(self, name, n, dtype):
        a = torch.empty(n + 2 * PAD, dtype=dtype, device="cuda")
        self._raw(a).fill_(self._canary(dtype))
        self.all[name] = a
        return a[PAD:PAD + n]

    @staticmethod
    def _raw(a):
        return a.view({torch.float32: torch.int32, torch.bfloat16: torch.int16, torch.uint8: torch.uint8}[a.dtype])

    @staticmethod
    def _canary(dtype):
        return {torch.float32: C32, torch.bfloat16: C16, torch.uint8: C8}[dtype]

    def check(self):
        torch.cuda.synchronize()
        for name, a in self.all.items():
            raw, c = self._raw(a), self._canary(a.dtype)
            assert (raw[:PAD] == c).all() and (raw[-PAD:] == c).all(), f"{name}: a write outside the buffer"


def W(name, shapes, units, N, mode, dtype):
    return synth.Workload(name, 41, list(shapes), list(units), N, mode, dtype, dtype, 2, 1e-3)


LAYOUTS = [
    W("aligned_dim0", [(512, 64), (64, 32), (256, 8)], [0, 0, 0], 4, synth.DIM0, torch.bfloat16),
    W("misaligned_flat", [(37, 5), (3,), (11, 13)], [0, 1, 1], 6, synth.FLAT, torch.bfloat16),
    W("fp32_groups", [(3000,), (129,)], [0, 0], 12, synth.FLAT, torch.float32),
]


@pytest.mark.parametrize("kind", ["auto", "direct", "staged"])
@pytest.mark.parametrize("w", LAYOUTS, ids=lambda w: w.name)
def test_no_write_outside_any_buffer(oracle_lib, w, kind):
    prev = fs.fsdp_set_rs_kernel(kind)
    try:
        _run(w)
    finally:
        fs.fsdp_set_rs_kernel(prev)


def _run(w):
    A = Arenas()
    L = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode)
    N, stride, F = w.N, L.stride, L.info["full_numel"]
    bf16 = w.param_dtype == torch.bfloat16
    O = pu.oracle_offsets(w)
    full32 = synth.full_params(w, F, O["t_full_off"])
    master, m, v = (A.make(k, N * stride, torch.float32) for k in ("master", "exp_avg", "exp_avg_sq"))
    gout = A.make("grad_out", N * stride, torch.float32)
    param = A.make("param", N * stride, torch.bfloat16) if bf16 else None
    full = A.make("full", F, w.param_dtype)
    fs.fsdp_reshard(L, 0, L.n_units, full32, master, param)
    m.zero_()
    v.zero_()
    for t in (1, 2):
        grads = synth.grad_replicas(w, F, t)
        fs.fsdp_unshard(L, 0, L.n_units, param if bf16 else master, full)
        fs.fsdp_reduce_scatter_adamw(L, 0, L.n_units, grads, master, m, v, param, gout, w.hp, t)
    # the sharded clip: the workspace and the norm output guarded too
    ws = A.make("clip_workspace", fs.fsdp_clip_workspace_bytes(), torch.uint8)
    norm = A.make("norm_out", 2, torch.float32)
    for t in (3, 4):
        grads = synth.grad_replicas(w, F, t)
        fs.fsdp_reduce_scatter_clip_adamw(L, 0, L.n_units, grads, master, m, v, param, gout, 1e-3, ws, norm, w.hp, t)
    # accumulation into guarded fp32 accumulators
    acc = [A.make(f"acc{q}", F, torch.float32) for q in range(N)]
    for mi in range(2):
        fs.fsdp_accumulate_grads(L, 0, L.n_units, acc, synth.grad_replicas(w, F, 10 + mi), first=(mi == 0))
    # the last micro-batch fused with the step, reading the guarded accumulators
    fs.fsdp_accumulate_reduce_scatter_adamw(L, 0, L.n_units, acc, synth.grad_replicas(w, F, 12), master, m, v, param,
                                            gout, w.hp, 5)
    # HSDP with two replica groups (the staged kernel may refuse a layout: then nothing runs)
    R = 2
    hm = A.make("hsdp_master", R * N * stride, torch.float32)
    hmm, hv = A.make("hsdp_m", R * N * stride, torch.float32), A.make("hsdp_v", R * N * stride, torch.float32)
    hp16 = A.make("hsdp_param", R * N * stride, torch.bfloat16) if bf16 else None
    # copy 0 is resharded (its base is aligned), the others start from the same shards;
    # a copy rho > 0 may begin off a 16-byte boundary, which the HSDP call accepts
    fs.fsdp_reshard(L, 0, L.n_units, full32, hm[:N * stride], hp16[:N * stride] if bf16 else None)
    for rho in range(1, R):
        hm[rho * N * stride:(rho + 1) * N * stride].copy_(hm[:N * stride])
        if bf16:
            hp16[rho * N * stride:(rho + 1) * N * stride].copy_(hp16[:N * stride])
    hmm.zero_()
    hv.zero_()
    try:
        fs.fsdp_hsdp_reduce_scatter_adamw(L, 0, L.n_units, R, [synth.grad_replica(w, F, 1, k) for k in range(R * N)],
                                          hm, hmm, hv, hp16, w.hp, 1)
    except fs.FsdpError as e:
        assert e.status == -1
    # ZeRO-1: guarded replicas and owner rows
    Z = fs.Layout(w.shapes, None, N, fs.FSDP_ZERO1)
    P = Z.info["numel"]
    zfull = synth.full_params(w, P, [Z.tensor(t)["full_off"] for t in range(len(w.shapes))])
    reps = [A.make(f"replica{q}", P, w.param_dtype) for q in range(N)]
    for r in reps:
        r.copy_(zfull.to(w.param_dtype))
    zm, zv = A.make("zero1_m", N * Z.stride, torch.float32), A.make("zero1_v", N * Z.stride, torch.float32)
    zm.zero_()
    zv.zero_()
    zmaster = A.make("zero1_master", N * Z.stride, torch.float32) if bf16 else None
    if bf16:
        fs.fsdp_reshard(Z, 0, Z.n_units, zfull, zmaster, None)
    try:
        fs.fsdp_zero1_adamw_broadcast(Z, 0, Z.n_units, synth.grad_replicas(w, P, 20), zmaster, zm, zv, reps, w.hp, 1)
    except fs.FsdpError as e:
        assert e.status == -1
    fs.fsdp_check_status()
    A.check()
