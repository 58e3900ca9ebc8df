"""Seeded random layouts (GPU): the staged and the direct kernels of every call
that has both (the fused step, HSDP, accumulation, ZeRO-1) must agree bit for
bit, and every fifth layout of the fused step is also compared with the oracle
element by element.

The layouts mix FLAT and DIM0 units, odd and empty tensors, row counts below N,
1..64 ranks, bf16 and fp32, so that pieces of both alignment classes, ragged
tile tails and replica groups (bf16 N > 16, fp32 N > 8) all occur.
"""
import numpy as np
import pytest
import torch

import fsdp_sharded_state_gb300 as fs
from fsdp_sharded_state_gb300 import synth

import parity_util as pu

pytestmark = pytest.mark.gpu


def random_workload(seed: int) -> synth.Workload:
    rng = np.random.default_rng(seed)
    mode = synth.FLAT if rng.random() < 0.6 else synth.DIM0
    N = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 12, 16, 24, 32, 64]))
    n_t = int(rng.integers(1, 7))
    shapes, units = [], []
    u = 0
    for t in range(n_t):
        kind = rng.random()
        if kind < 0.15:
            s = (int(rng.integers(0, 3)), int(rng.integers(0, 9)))        # tiny or empty
        elif kind < 0.3:
            s = (int(rng.integers(1, 5000)),)                           # 1-D
        elif kind < 0.45:
            s = ()                                                      # scalar
        else:
            s = (int(rng.integers(1, 700)), int(rng.integers(1, 300)))
        shapes.append(s)
        if t > 0 and rng.random() < 0.4:
            u += 1
        units.append(u)
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    return synth.Workload(f"random{seed}", 20, shapes, units, N, mode, dtype, dtype, 2, 1e-3)


def run(w, kind, strategy):
    prev = fs.fsdp_set_rs_kernel(kind)
    try:
        O = pu.oracle_offsets(w)
        st = pu.make_state(w, with_grad_out=True)
        st.init_from_full(synth.full_params(w, O["F"], O["t_full_off"], device="cuda"))
        for t in range(1, w.steps + 1):
            st.step(synth.grad_replicas(w, O["F"], t, device="cuda"), w.hp, strategy=strategy)
        torch.cuda.synchronize()
        return st
    finally:
        fs.fsdp_set_rs_kernel(prev)


@pytest.mark.parametrize("seed", list(range(40)))
def test_staged_equals_direct_on_random_layouts(oracle_lib, seed):
    w = random_workload(seed)
    strategy = "full_shard" if seed % 2 else "shard_grad_op"
    a = run(w, "direct", strategy)
    b = run(w, "staged", strategy)
    for name in ("master", "exp_avg", "exp_avg_sq", "grad_out"):
        assert torch.equal(getattr(a, name).view(torch.int32), getattr(b, name).view(torch.int32)), (name, w.shapes, w.N)
    if a.param is not None:
        assert torch.equal(a.param.view(torch.int16), b.param.view(torch.int16)), ("param", w.shapes, w.N)
    assert torch.equal(a.full.view(torch.int16 if a.full.dtype == torch.bfloat16 else torch.int32),
                       b.full.view(torch.int16 if b.full.dtype == torch.bfloat16 else torch.int32))
    if seed % 5 == 0:
        pu.run_full_parity(w, strategy=strategy)


def run_rows(w, kind, R):
    """HSDP (R groups), accumulation (3 micro-batches) and ZeRO-1 on the same layout."""
    prev = fs.fsdp_set_rs_kernel(kind)
    try:
        L = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode)
        F, stride, N = L.info["full_numel"], L.stride, w.N
        O = pu.oracle_offsets(w)
        full = synth.full_params(w, F, O["t_full_off"], device="cuda")
        bf16 = w.param_dtype == torch.bfloat16
        out = {}
        master = torch.zeros(R, N, stride, dtype=torch.float32, device="cuda")
        param = torch.zeros(R, N, stride, dtype=torch.bfloat16, device="cuda") if bf16 else None
        fs.fsdp_reshard(L, 0, L.n_units, full, master[0], param[0] if bf16 else None)
        for rho in range(1, R):
            master[rho].copy_(master[0])
            if bf16:
                param[rho].copy_(param[0])
        m, v = torch.zeros_like(master), torch.zeros_like(master)
        grads = [synth.grad_replica(w, F, 1, rho * N + q) for rho in range(R) for q in range(N)]
        try:
            fs.fsdp_hsdp_reduce_scatter_adamw(L, 0, L.n_units, R, grads, master, m, v, param, w.hp, 1)
            out["hsdp"] = (master, m, v, param)
        except fs.FsdpError as e:
            if not (kind == "staged" and e.status == -1):      # the staged HSDP kernel does not hold it
                raise
        acc = [torch.zeros(F, dtype=torch.float32, device="cuda") for _ in range(N)]
        for mi in range(3):
            micro = synth.grad_replicas(w, F, 10 + mi)
            fs.fsdp_accumulate_grads(L, 0, L.n_units, acc, micro, first=(mi == 0))
        out["acc"] = acc
        # ZeRO-1 on the same tensors
        Z = fs.Layout(w.shapes, None, N, fs.FSDP_ZERO1)
        P = Z.info["numel"]
        zoffs = [Z.tensor(t)["full_off"] for t in range(len(w.shapes))]
        zfull = synth.full_params(w, P, zoffs, device="cuda")
        reps = [zfull.to(w.param_dtype).clone() for _ in range(N)]
        zmaster = torch.zeros(N, Z.stride, dtype=torch.float32, device="cuda") if bf16 else None
        if bf16:
            fs.fsdp_reshard(Z, 0, Z.n_units, zfull, zmaster, None)
        zm = torch.zeros(N, Z.stride, dtype=torch.float32, device="cuda")
        zv = torch.zeros_like(zm)
        try:
            for t in range(1, 3):
                fs.fsdp_zero1_adamw_broadcast(Z, 0, Z.n_units, synth.grad_replicas(w, P, 20 + t), zmaster, zm, zv,
                                              reps, w.hp, t)
            out["zero1"] = reps + [zm, zv] + ([zmaster] if bf16 else [])
        except fs.FsdpError as e:
            if not (kind == "staged" and e.status == -1):      # the staged ZeRO-1 kernel does not hold it
                raise
        torch.cuda.synchronize()
        return out
    finally:
        fs.fsdp_set_rs_kernel(prev)


@pytest.mark.parametrize("seed", list(range(0, 40, 2)))
def test_staged_rows_equal_direct_on_random_layouts(seed):
    w = random_workload(seed)
    if w.N > 16:
        w.N = 16                     # R * N <= 64 replicas for the HSDP call
    R = 2 + (seed // 2) % 2
    a = run_rows(w, "direct", R)
    b = run_rows(w, "staged", R)
    if "hsdp" in b:
        for x, y in zip(a["hsdp"], b["hsdp"]):
            if x is not None:
                assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x.view(torch.int16),
                                   y.view(torch.int32) if y.dtype == torch.float32 else y.view(torch.int16))
    for x, y in zip(a["acc"], b["acc"]):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    for x, y in zip(a["zero1"], b.get("zero1", a["zero1"])):
        assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x.view(torch.int16),
                           y.view(torch.int32) if y.dtype == torch.float32 else y.view(torch.int16))
