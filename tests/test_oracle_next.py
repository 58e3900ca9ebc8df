"""Pins of the oracle's rows beyond the core step (CPU): sharded clip_grad_norm_,
gradient accumulation without sync, HSDP and the ZeRO-1 owner partition.

Each is checked against torch's own implementation on gloo CPU ranks (FSDP1
clip_grad_norm_ and no_sync, FSDP2 fully_shard on a 2-D mesh, the
ZeroRedundancyOptimizer) and against invariants that follow from the pages.
"""
import os
import sys

import numpy as np
import pytest
import torch

import oracle
from test_oracle_torch_fsdp import free_port, pack_full, WORKER

import subprocess

HP = (1e-3, 0.9, 0.999, 1e-8, 0.01)


def run_worker(tmp_path, mode, n, shapes, steps=3, R=1, clip=0.0, accum=1, seed=1):
    spec = ",".join("x".join(str(d) for d in s) if s else "scalar" for s in shapes)
    cmd = [sys.executable, WORKER, "--mode", mode, "--n", str(n), "--R", str(R), "--shapes", spec,
           "--steps", str(steps), "--seed", str(seed), "--clip", str(clip), "--accum", str(accum),
           "--port", str(free_port()), "--out", str(tmp_path)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=dict(os.environ, OMP_NUM_THREADS="1"))
    assert r.returncode == 0, r.stderr[-3000:]
    return [torch.load(os.path.join(tmp_path, f"rank{k}.pt")) for k in range(n * R)]


def band(got, ref, rel=1e-5, atol=1e-8):
    err = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    assert (err <= rel * np.abs(ref) + atol).all(), err.max()


def logical_mask(L, shapes):
    mask = np.zeros(L["F"], bool)
    for t, s in enumerate(shapes):
        mask[L["t_full_off"][t]:L["t_full_off"][t] + int(np.prod(s) if s else 1)] = True
    return mask


# ---------------------------------------------------------------------------
# sharded clip_grad_norm_
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode,n,shapes,clip", [
    ("flat", 3, [(5, 3), (4,)], 1e-3),        # clipping active (norm ~ 4e-3)
    ("flat", 3, [(5, 3), (4,)], 10.0),        # not active: coefficient 1
    ("dim0", 3, [(5, 3), (7,), (2, 4)], 1e-3),
])
def test_clip_matches_torch_fsdp(oracle_lib, tmp_path, mode, n, shapes, clip):
    outs = run_worker(tmp_path, mode, n, shapes, steps=3, clip=clip)
    om = oracle.FLAT if mode == "flat" else oracle.DIM0
    sh = oracle.Shapes(shapes)
    L = oracle.layout(sh, n, om)
    stride = L["S"]
    master, _ = oracle.reshard(sh, n, om, pack_full(L, outs[0]["init"]), stride, True, False)
    m, v, gout = np.zeros_like(master), np.zeros_like(master), np.zeros_like(master)
    for t in range(3):
        grads = [pack_full(L, outs[r]["grads"][t][0]) for r in range(n)]
        norm = oracle.rs_clip_adamw(sh, n, om, grads, stride, master, m, v, clip, grad_out=gout, hp=HP, step=t + 1)
        assert norm == pytest.approx(outs[0]["norms"][t], rel=1e-5)
        for r in range(n):
            row = gout[r * stride:(r + 1) * stride]
            if om == oracle.FLAT:
                band(outs[r]["grad_shards"][t][0].numpy(), row[:L["S"]], 2e-6, 2e-10)
            else:
                for k in range(len(shapes)):
                    got = outs[r]["grad_shards"][t][k].numpy().reshape(-1)
                    o = L["t_shard_off"][k]
                    band(got, row[o:o + got.size], 2e-6, 2e-10)
    mask = logical_mask(L, shapes)
    band(oracle.unshard(sh, n, om, master, stride, L["F"])[mask], pack_full(L, outs[0]["final"])[mask])


def test_clip_closed_forms(oracle_lib):
    sh = oracle.Shapes([(7, 5), (9,)])
    N = 4
    L = oracle.layout(sh, N, oracle.FLAT)
    rng = np.random.default_rng(2)
    full = rng.normal(0, 0.02, L["F"]).astype(np.float32)
    grads = [rng.normal(0, 1e-2, L["F"]).astype(np.float32) for _ in range(N)]
    # the norm is that of the averaged full gradient (single-rank clip equivalence)
    mean = np.zeros(L["F"])
    for g in grads:
        mean += g.astype(np.float64)
    mean /= N
    mask = logical_mask(L, [(7, 5), (9,)])
    ref_norm = float(np.sqrt((mean[mask] ** 2).sum()))
    a_m, _ = oracle.reshard(sh, N, oracle.FLAT, full, L["S"], True, False)
    b_m = a_m.copy()
    z = lambda: np.zeros_like(a_m)
    ma, va, mb, vb, gout = z(), z(), z(), z(), z()
    norm = oracle.rs_clip_adamw(sh, N, oracle.FLAT, grads, L["S"], a_m, ma, va, 1e9, hp=HP, step=1)
    assert norm == pytest.approx(ref_norm, rel=1e-6)
    # max_norm far above the norm: coefficient 1, the plain step bit for bit
    oracle.rs_adamw(sh, N, oracle.FLAT, grads, L["S"], b_m, mb, vb, hp=HP, step=1)
    assert np.array_equal(a_m.view(np.uint32), b_m.view(np.uint32))
    # active clipping: the clipped gradient's norm is max_norm * norm / (norm + 1e-6)
    c_m, _ = oracle.reshard(sh, N, oracle.FLAT, full, L["S"], True, False)
    mx = ref_norm / 4
    oracle.rs_clip_adamw(sh, N, oracle.FLAT, grads, L["S"], c_m, z(), z(), mx, grad_out=gout, hp=HP, step=1)
    assert float(np.sqrt((gout.astype(np.float64) ** 2).sum())) == pytest.approx(mx * ref_norm / (ref_norm + 1e-6),
                                                                                rel=2e-7)


def test_clip_matches_torch_clip_grad_norm(oracle_lib):
    # library routine: torch.nn.utils.clip_grad_norm_ on the averaged full gradient
    shapes = [(11, 6), (13,)]
    sh = oracle.Shapes(shapes)
    N = 4
    L = oracle.layout(sh, N, oracle.FLAT)
    rng = np.random.default_rng(5)
    full = rng.normal(0, 0.02, L["F"]).astype(np.float32)
    grads = [rng.normal(0, 1e-2, L["F"]).astype(np.float32) for _ in range(N)]
    master, _ = oracle.reshard(sh, N, oracle.FLAT, full, L["S"], True, False)
    gout = np.zeros_like(master)
    norm = oracle.rs_clip_adamw(sh, N, oracle.FLAT, grads, L["S"], master, np.zeros_like(master),
                                np.zeros_like(master), 0.01, grad_out=gout, hp=HP, step=1)
    mask = logical_mask(L, shapes)
    ps = []
    for t, s in enumerate(shapes):
        o, k = L["t_full_off"][t], int(np.prod(s))
        p = torch.nn.Parameter(torch.zeros(k))
        p.grad = torch.from_numpy(np.mean([g[o:o + k] for g in grads], axis=0).astype(np.float32))
        ps.append(p)
    tn = torch.nn.utils.clip_grad_norm_(ps, 0.01)
    assert float(tn) == pytest.approx(norm, rel=1e-6)
    got = oracle.unshard(sh, N, oracle.FLAT, gout, L["S"], L["F"])
    ref = np.zeros(L["F"], np.float32)
    for t, p in enumerate(ps):
        ref[L["t_full_off"][t]:L["t_full_off"][t] + p.numel()] = p.grad.numpy()
    band(got[mask], ref[mask], 1e-6, 1e-12)


# ---------------------------------------------------------------------------
# gradient accumulation without sync
# ---------------------------------------------------------------------------
def test_accumulation_matches_torch_no_sync(oracle_lib, tmp_path):
    shapes, n, M = [(5, 3), (4,)], 3, 3
    outs = run_worker(tmp_path, "flat", n, shapes, steps=2, accum=M)
    sh = oracle.Shapes(shapes)
    L = oracle.layout(sh, n, oracle.FLAT)
    stride = L["S"]
    master, _ = oracle.reshard(sh, n, oracle.FLAT, pack_full(L, outs[0]["init"]), stride, True, False)
    m, v, gout = np.zeros_like(master), np.zeros_like(master), np.zeros_like(master)
    for t in range(2):
        accs = [np.zeros(L["F"], np.float32) for _ in range(n)]
        for mi in range(M):
            for r in range(n):
                oracle.accumulate(accs[r], pack_full(L, outs[r]["grads"][t][mi]), first=(mi == 0))
        oracle.rs_adamw(sh, n, oracle.FLAT, accs, stride, master, m, v, grad_out=gout, hp=HP, step=t + 1)
        for r in range(n):
            band(outs[r]["grad_shards"][t][0].numpy(), gout[r * stride:r * stride + L["S"]], 2e-6, 2e-10)
    mask = logical_mask(L, shapes)
    band(oracle.unshard(sh, n, oracle.FLAT, master, stride, L["F"])[mask], pack_full(L, outs[0]["final"])[mask])


def test_accumulation_closed_form(oracle_lib):
    # accumulating M micro-gradients per replica, then one reduce-scatter, is the
    # reduce-scatter of the per-replica sums (same order: micro then rank)
    rng = np.random.default_rng(8)
    n, M = 4, 5
    micro = [[rng.normal(0, 1e-3, 50).astype(np.float32) for _ in range(M)] for _ in range(n)]
    accs = []
    for r in range(n):
        a = np.zeros(50, np.float32)
        for mi in range(M):
            oracle.accumulate(a, micro[r][mi], first=(mi == 0))
        s = micro[r][0].copy()
        for mi in range(1, M):
            s = (s + micro[r][mi]).astype(np.float32)
        assert np.array_equal(a.view(np.uint32), s.view(np.uint32))
        accs.append(a)


# ---------------------------------------------------------------------------
# HSDP
# ---------------------------------------------------------------------------
def test_hsdp_matches_torch_2d_mesh(oracle_lib, tmp_path):
    shapes, n, R = [(5, 3), (7,), (2, 4)], 2, 2
    outs = run_worker(tmp_path, "hsdp", n, shapes, steps=3, R=R)
    sh = oracle.Shapes(shapes)
    L = oracle.layout(sh, n, oracle.DIM0)
    stride = L["S"]
    m0, _ = oracle.reshard(sh, n, oracle.DIM0, pack_full(L, outs[0]["init"]), stride, True, False)
    master = np.concatenate([m0] * R)
    m, v = np.zeros_like(master), np.zeros_like(master)
    for t in range(3):
        # mesh rank order: global rank = rho * n + q
        grads = [pack_full(L, outs[rho * n + q]["grads"][t][0]) for rho in range(R) for q in range(n)]
        oracle.hsdp_adamw(sh, n, oracle.DIM0, R, grads, stride, master, m, v, hp=HP, step=t + 1)
    mask = logical_mask(L, shapes)
    final = pack_full(L, outs[0]["final"])
    for rho in range(R):
        got = oracle.unshard(sh, n, oracle.DIM0, master[rho * n * stride:(rho + 1) * n * stride], stride, L["F"])
        band(got[mask], final[mask])


def test_hsdp_reductions(oracle_lib):
    # R = 1 is the plain sharded step; any R matches DDP over R*N ranks (up to order)
    shapes = [(9, 4), (5,)]
    sh = oracle.Shapes(shapes)
    N = 3
    L = oracle.layout(sh, N, oracle.FLAT)
    rng = np.random.default_rng(4)
    full = rng.normal(0, 0.02, L["F"]).astype(np.float32)
    m0, _ = oracle.reshard(sh, N, oracle.FLAT, full, L["S"], True, False)
    g = [rng.normal(0, 1e-3, L["F"]).astype(np.float32) for _ in range(2 * N)]
    a = m0.copy()
    oracle.hsdp_adamw(sh, N, oracle.FLAT, 1, g[:N], L["S"], a, np.zeros_like(a), np.zeros_like(a), hp=HP, step=1)
    b = m0.copy()
    oracle.rs_adamw(sh, N, oracle.FLAT, g[:N], L["S"], b, np.zeros_like(b), np.zeros_like(b), hp=HP, step=1)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    c = np.concatenate([m0, m0])
    oracle.hsdp_adamw(sh, N, oracle.FLAT, 2, g, L["S"], c, np.zeros_like(c), np.zeros_like(c), hp=HP, step=1)
    assert np.array_equal(c[:N * L["S"]].view(np.uint32), c[N * L["S"]:].view(np.uint32))   # groups agree
    mask = logical_mask(L, shapes)
    p = full.copy()
    oracle.ddp_adamw(g, p, np.zeros_like(p), np.zeros_like(p), skip=~mask, hp=HP, step=1)
    band(oracle.unshard(sh, N, oracle.FLAT, c[:N * L["S"]], L["S"], L["F"])[mask], p[mask], 1e-6, 1e-9)


# ---------------------------------------------------------------------------
# ZeRO-1
# ---------------------------------------------------------------------------
ZSHAPES = [(7, 5), (3,), (9, 2), (4, 4), (11,), (6, 6)]


def test_zero1_owners_and_result_match_torch_zro(oracle_lib, tmp_path):
    n = 3
    outs = run_worker(tmp_path, "zero1", n, ZSHAPES, steps=3)
    sh = oracle.Shapes(ZSHAPES)
    owners = oracle.zero1_owners(sh, n)
    for r in range(n):
        assert [o == r for o in owners] == outs[r]["owners_mine"], r
    sizes = [int(np.prod(s)) for s in ZSHAPES]
    stride = max(sum(sz for sz, o in zip(sizes, owners) if o == r) for r in range(n))
    P = sum(sizes)
    init = np.concatenate([x.numpy().reshape(-1) for x in outs[0]["init"]]).astype(np.float32)
    params = [init.copy() for _ in range(n)]
    m = np.zeros(n * stride, np.float32)
    v = np.zeros(n * stride, np.float32)
    for t in range(3):
        grads = [np.concatenate([x.numpy().reshape(-1) for x in outs[r]["grads"][t][0]]).astype(np.float32)
                 for r in range(n)]
        params = oracle.zero1_adamw(sh, n, grads, stride, None, m, v, params, hp=HP, step=t + 1)
    final = np.concatenate([x.numpy().reshape(-1) for x in outs[0]["final"]])
    for q in range(n):
        band(params[q], final)
    assert P == init.size


def test_zero1_equals_ddp_bitwise(oracle_lib):
    # every parameter is updated once, by its owner, with the averaged gradient and
    # the same AdamW: the replicated (ZeRO-0) result bit for bit, on every replica
    n = 4
    sh = oracle.Shapes(ZSHAPES)
    rng = np.random.default_rng(6)
    P = sum(int(np.prod(s)) for s in ZSHAPES)
    init = rng.normal(0, 0.02, P).astype(np.float32)
    owners = oracle.zero1_owners(sh, n)
    sizes = [int(np.prod(s)) for s in ZSHAPES]
    stride = max(sum(sz for sz, o in zip(sizes, owners) if o == r) for r in range(n))
    params = [init.copy() for _ in range(n)]
    master = np.zeros(n * stride, np.float32)
    m, v = np.zeros_like(master), np.zeros_like(master)
    p, pm, pv = init.copy(), np.zeros(P, np.float32), np.zeros(P, np.float32)
    for t in range(1, 4):
        grads = [rng.normal(0, 1e-3, P).astype(np.float32) for _ in range(n)]
        params = oracle.zero1_adamw(sh, n, grads, stride, None, m, v, params, hp=HP, step=t)
        oracle.ddp_adamw(grads, p, pm, pv, hp=HP, step=t)
    for q in range(n):
        assert np.array_equal(params[q].view(np.uint32), p.view(np.uint32))


def test_zero1_owner_balance_by_size(oracle_lib):
    # byte balance, not parameter-count balance: one big tensor and many small ones
    sh = oracle.Shapes([(1000,)] + [(10,)] * 9)
    owners = oracle.zero1_owners(sh, 2)
    assert owners[0] == 0 and all(o == 1 for o in owners[1:])
