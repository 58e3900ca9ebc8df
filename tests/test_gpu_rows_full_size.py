"""The rows beyond the core step at the size bench.py times them (GPU): the 128 MiB
fp32 layout (8 x [2048,2048], N = 4), every element against the oracle.

  clip   fsdp_reduce_scatter_clip_adamw with max_norm 1e-2 (the bench's call; the clip
         is active), two steps: clipped gradient shard, master, moments, norm.
  accum  fsdp_accumulate_grads over three micro-batches: every accumulator element.
  hsdp   fsdp_hsdp_reduce_scatter_adamw with R = 2 groups, two steps: both state copies.
  zero1  fsdp_zero1_adamw_broadcast with fp32 replicas, two steps: every replica and the
         owners' moments.
Each with the automatic kernel choice, the launch configuration the bench times.
"""
import numpy as np
import pytest
import torch

import fsdp_sharded_state_gb300 as fs
import oracle
from fsdp_sharded_state_gb300 import synth

import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture
def w():
    return synth.mlp128m()


def test_clip_at_bench_size(oracle_lib, w):
    st = pu.make_state(w, with_grad_out=True)
    sh = oracle.Shapes(w.shapes, w.unit_ids)
    O = pu.oracle_offsets(w)
    full = synth.full_params(w, st.F, O["t_full_off"])
    st.init_from_full(full)
    om, _ = oracle.reshard(sh, w.N, w.mode, pu.f32(full), st.stride, True, False)
    m, v, go = np.zeros_like(om), np.zeros_like(om), np.zeros_like(om)
    ws = torch.empty(fs.fsdp_clip_workspace_bytes(), dtype=torch.uint8, device="cuda")
    norm_out = torch.zeros(2, dtype=torch.float32, device="cuda")
    for t in (1, 2):
        grads = synth.grad_replicas(w, st.F, t)
        fs.fsdp_reduce_scatter_clip_adamw(st.layout, 0, st.layout.n_units, grads, st.master, st.exp_avg,
                                          st.exp_avg_sq, None, st.grad_out, 1e-2, ws, norm_out, w.hp, t)
        ref = oracle.rs_clip_adamw(sh, w.N, w.mode, pu.grads_np(grads), st.stride, om, m, v, 1e-2, grad_out=go,
                                   hp=w.hp, step=t)
        torch.cuda.synchronize()
        got_norm, got_coef = norm_out.tolist()
        assert got_norm == pytest.approx(ref, rel=1e-6)
        assert got_coef < 1.0                          # the clip is active at this size
        for x, y, what in ((st.grad_out, go, "clipped grad"), (st.master, om, "master"), (st.exp_avg, m, "exp_avg"),
                           (st.exp_avg_sq, v, "exp_avg_sq")):
            pu.assert_f32_close(pu.f32(x).reshape(-1), y, f"{what} step {t}")


def test_accumulate_at_bench_size(oracle_lib, w):
    L = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode)
    F = L.info["full_numel"]
    acc = [torch.zeros(F, dtype=torch.float32, device="cuda") for _ in range(w.N)]
    ref = [np.zeros(F, np.float32) for _ in range(w.N)]
    for mi in range(3):
        micro = synth.grad_replicas(w, F, 10 + mi)
        fs.fsdp_accumulate_grads(L, 0, L.n_units, acc, micro, first=(mi == 0))
        for q, g in enumerate(pu.grads_np(micro)):
            oracle.accumulate(ref[q], g, first=(mi == 0))
    torch.cuda.synchronize()
    for q in range(w.N):                               # no padding in this layout: every element
        assert np.array_equal(pu.f32(acc[q]).view(np.uint32), ref[q].view(np.uint32)), f"accumulator {q}"


def test_hsdp_at_bench_size(oracle_lib, w):
    R, N = 2, w.N
    L = fs.Layout(w.shapes, w.unit_ids, N, w.mode)
    sh = oracle.Shapes(w.shapes, w.unit_ids)
    O = pu.oracle_offsets(w)
    stride, F = L.stride, L.info["full_numel"]
    full = synth.full_params(w, F, O["t_full_off"])
    master = torch.zeros(R, N, stride, dtype=torch.float32, device="cuda")
    fs.fsdp_reshard(L, 0, L.n_units, full, master[0], None)
    master[1].copy_(master[0])
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    om1, _ = oracle.reshard(sh, N, w.mode, pu.f32(full), stride, True, False)
    om = np.concatenate([om1] * R)
    rm, rv = np.zeros_like(om), np.zeros_like(om)
    for t in (1, 2):
        grads = [synth.grad_replica(w, F, t, k) for k in range(R * N)]
        fs.fsdp_hsdp_reduce_scatter_adamw(L, 0, L.n_units, R, grads, master, m, v, None, w.hp, t)
        oracle.hsdp_adamw(sh, N, w.mode, R, pu.grads_np(grads), stride, om, rm, rv, hp=w.hp, step=t)
        torch.cuda.synchronize()
        for x, y, what in ((master, om, "master"), (m, rm, "exp_avg"), (v, rv, "exp_avg_sq")):
            pu.assert_f32_close(pu.f32(x).reshape(-1), y, f"hsdp {what} step {t}")


def test_zero1_at_bench_size(oracle_lib, w):
    N = w.N
    L = fs.Layout(w.shapes, None, N, fs.FSDP_ZERO1)
    sh = oracle.Shapes(w.shapes)
    owners = oracle.zero1_owners(sh, N)
    P = L.info["numel"]
    offs = [L.tensor(t)["full_off"] for t in range(len(w.shapes))]
    full = synth.full_params(w, P, offs)
    params = [full.clone() for _ in range(N)]
    m = torch.zeros(N, L.stride, dtype=torch.float32, device="cuda")
    v = torch.zeros_like(m)
    ooff, ostride = pu.oracle_zero1_rows(sh, N, owners)
    rm = np.zeros(N * ostride, np.float32)
    rv = np.zeros_like(rm)
    rparams = [pu.f32(full) for _ in range(N)]
    for t in (1, 2):
        grads = synth.grad_replicas(w, P, t)
        fs.fsdp_zero1_adamw_broadcast(L, 0, L.n_units, grads, None, m, v, params, w.hp, t)
        rparams = oracle.zero1_adamw(sh, N, pu.grads_np(grads), ostride, None, rm, rv, rparams, hp=w.hp, step=t)
        torch.cuda.synchronize()
        for q in range(N):
            pu.assert_f32_close(pu.f32(params[q]), rparams[q], f"replica {q} step {t}")
        gm, gv = pu.f32(m).reshape(-1), pu.f32(v).reshape(-1)
        n = 2048 * 2048
        for k, o in enumerate(owners):
            a = o * L.stride + L.tensor(k)["shard_off"]
            b = o * ostride + ooff[k]
            pu.assert_f32_close(gm[a:a + n], rm[b:b + n], f"exp_avg t{k} step {t}")
            pu.assert_f32_close(gv[a:a + n], rv[b:b + n], f"exp_avg_sq t{k} step {t}")
