"""Seeded random layouts (GPU): the staged and the direct kernels of every call
that has both (the fused step, HSDP, accumulation, ZeRO-1) must agree bit for
bit, and every fifth layout of the fused step, and every fifth layout of the
rows (HSDP, accumulation, ZeRO-1), is also compared with the oracle element by
element.

The layouts mix FLAT and DIM0 units, odd and empty tensors, row counts below N,
1..64 ranks, bf16 and fp32, so that pieces of both alignment classes, ragged
tile tails and replica groups (bf16 N > 16, fp32 N > 8) all occur.
"""
import numpy as np
import pytest
import torch

import fsdp_sharded_state_gb300 as fs
import oracle
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


def _bits(x):
    return x.view(torch.int32) if x.dtype == torch.float32 else x.view(torch.int16)


_ROWS_CACHE = {}


def rows_runs(seed):
    """The layout of `seed`, its R, and the direct and staged runs of its rows (kept for
    the three row tests of the seed; only the latest seed is held)."""
    if seed not in _ROWS_CACHE:
        _ROWS_CACHE.clear()
        w = random_workload(seed)
        if w.N > 16:
            w.N = 16                 # R * N <= 64 replicas for the HSDP call
        R = 2 + (seed // 2) % 2
        _ROWS_CACHE[seed] = (w, R, run_rows(w, "direct", R), run_rows(w, "staged", R))
    return _ROWS_CACHE[seed]


@pytest.mark.parametrize("row", ["hsdp", "acc", "zero1"])
@pytest.mark.parametrize("seed", list(range(0, 40, 2)))
def test_staged_rows_equal_direct_on_random_layouts(oracle_lib, seed, row):
    w, R, a, b = rows_runs(seed)
    if (seed // 2) % 5 == 0:         # every fifth layout: the direct results against the oracle
        rows_vs_oracle(w, R, a, row)
    if row not in b:
        # the staged kernel does not hold this layout: the call refused it (FSDP_EINVAL)
        pytest.skip(f"staged {row} kernel refused the layout (N={w.N}, R={R}); nothing to compare")
    for x, y in zip(a[row], b[row]):
        if x is not None:
            assert torch.equal(_bits(x), _bits(y)), (row, w.shapes, w.N)


def rows_vs_oracle(w, R, out, row):
    """One row's results of run_rows (HSDP, accumulation or ZeRO-1) against the oracle,
    on the same seeded inputs."""
    sh = oracle.Shapes(w.shapes, w.unit_ids)
    O = pu.oracle_offsets(w)
    N, F = w.N, O["F"]
    stride = fs.Layout(w.shapes, w.unit_ids, N, w.mode).stride
    bf16 = w.param_dtype == torch.bfloat16
    full = pu.f32(synth.full_params(w, F, O["t_full_off"], device="cuda"))
    if row == "hsdp":
        return _hsdp_vs_oracle(w, R, out, sh, O, N, F, stride, bf16, full)
    if row == "acc":
        return _acc_vs_oracle(w, out, O, N, F)
    return _zero1_vs_oracle(w, out, N, bf16)


def _hsdp_vs_oracle(w, R, out, sh, O, N, F, stride, bf16, full):
    # R groups start from the same shards, one step
    om1, op1 = oracle.reshard(sh, N, w.mode, full, stride, True, bf16)
    om = np.concatenate([om1] * R)
    op = np.concatenate([op1] * R) if bf16 else None
    m, v = np.zeros_like(om), np.zeros_like(om)
    grads = [synth.grad_replica(w, F, 1, rho * N + q) for rho in range(R) for q in range(N)]
    oracle.hsdp_adamw(sh, N, w.mode, R, pu.grads_np(grads), stride, om, m, v, param=op, hp=w.hp, step=1)
    master, gm, gv, param = out["hsdp"]
    pu.assert_f32_close(pu.f32(master).reshape(-1), om, "hsdp master")
    pu.assert_f32_close(pu.f32(gm).reshape(-1), m, "hsdp exp_avg")
    pu.assert_f32_close(pu.f32(gv).reshape(-1), v, "hsdp exp_avg_sq")
    if bf16:
        pu.assert_bf16_close(pu.u16(param).reshape(-1), op, "hsdp param")


def _acc_vs_oracle(w, out, O, N, F):
    # 3 micro-batches, logical positions (FLAT padding is not touched)
    mask = pu.logical(O, w.shapes)
    ref = [np.zeros(F, np.float32) for _ in range(N)]
    for mi in range(3):
        micro = pu.grads_np(synth.grad_replicas(w, F, 10 + mi))
        for q in range(N):
            oracle.accumulate(ref[q], micro[q], first=(mi == 0))
    for q in range(N):
        assert np.array_equal(pu.f32(out["acc"][q])[mask].view(np.uint32), ref[q][mask].view(np.uint32)), f"acc {q}"


def _zero1_vs_oracle(w, out, N, bf16):
    # the same tensors in a ZeRO-1 layout, two steps
    zsh = oracle.Shapes(w.shapes)
    Z = fs.Layout(w.shapes, None, N, fs.FSDP_ZERO1)
    P = Z.info["numel"]
    zoffs = [Z.tensor(t)["full_off"] for t in range(len(w.shapes))]
    zfull = synth.full_params(w, P, zoffs, device="cuda")
    owners = oracle.zero1_owners(zsh, N)
    ooff, ostride = pu.oracle_zero1_rows(zsh, N, owners)
    sizes = [int(np.prod(s) if s else 1) for s in w.shapes]
    rm = np.zeros(N * max(ostride, 1), np.float32)
    rv = np.zeros_like(rm)
    rmaster = None
    f = pu.f32(zfull)
    if bf16:
        rmaster = np.zeros_like(rm)
        for t, o in enumerate(owners):
            rmaster[o * ostride + ooff[t]:o * ostride + ooff[t] + sizes[t]] = f[zoffs[t]:zoffs[t] + sizes[t]]
    rparams = [pu.u16(zfull.to(torch.bfloat16)) if bf16 else f.copy() for _ in range(N)]
    for t in range(1, 3):
        g = pu.grads_np(synth.grad_replicas(w, P, 20 + t))
        rparams = oracle.zero1_adamw(zsh, N, g, ostride, rmaster, rm, rv, rparams, hp=w.hp, step=t)
    reps, zm, zv = out["zero1"][:N], out["zero1"][N], out["zero1"][N + 1]
    for q in range(N):
        if bf16:
            pu.assert_bf16_close(pu.u16(reps[q]), rparams[q], f"zero1 replica {q}")
        else:
            pu.assert_f32_close(pu.f32(reps[q]), rparams[q], f"zero1 replica {q}")
    gm, gv = pu.f32(zm).reshape(-1), pu.f32(zv).reshape(-1)
    for k, o in enumerate(owners):
        a = o * Z.stride + Z.tensor(k)["shard_off"]
        b = o * ostride + ooff[k]
        pu.assert_f32_close(gm[a:a + sizes[k]], rm[b:b + sizes[k]], f"zero1 exp_avg t{k}")
        pu.assert_f32_close(gv[a:a + sizes[k]], rv[b:b + sizes[k]], f"zero1 exp_avg_sq t{k}")


# ---------------------------------------------------------------------------
# Large random layouts: hundreds of tensors (many small, some large), 3-8M parameters,
# so that a launch has thousands of tiles and its CTAs claim them from a counter, each
# claim jumping the CTA's segment cursor across many segments.  The staged kernels
# (claimed tiles) against the direct ones (a static split) bit for bit, and every other
# layout against the oracle.
def big_random_workload(seed: int) -> synth.Workload:
    rng = np.random.default_rng(7000 + seed)
    mode = synth.FLAT if seed % 2 == 0 else synth.DIM0
    N = int(rng.choice([2, 3, 4, 6, 8, 16]))
    shapes = [(int(rng.integers(1, 5000)),) if rng.random() < 0.5 else (int(rng.integers(1, 40)), int(rng.integers(1, 200)))
              for _ in range(int(rng.integers(100, 300)))]
    shapes += [(int(rng.integers(200, 2000)), int(rng.integers(64, 1024))) for _ in range(int(rng.integers(10, 30)))]
    order = rng.permutation(len(shapes))
    shapes = [shapes[i] for i in order]
    units, u = [], 0
    for t in range(len(shapes)):
        if t > 0 and rng.random() < 0.05:
            u += 1
        units.append(u)
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    return synth.Workload(f"bigrandom{seed}", 20, shapes, units, N, mode, dtype, dtype, 2, 1e-3)


@pytest.mark.parametrize("seed", list(range(6)))
def test_staged_equals_direct_on_large_random_layouts(oracle_lib, seed):
    w = big_random_workload(seed)
    L = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode)
    assert L.stride * w.N >= 8 * 152 * 2048          # enough tiles for the claims
    strategy = "full_shard"
    a = run(w, "direct", strategy)
    b = run(w, "staged", strategy)
    for name in ("master", "exp_avg", "exp_avg_sq", "grad_out"):
        assert torch.equal(getattr(a, name).view(torch.int32), getattr(b, name).view(torch.int32)), (name, w.N)
    if a.param is not None:
        assert torch.equal(a.param.view(torch.int16), b.param.view(torch.int16)), ("param", w.N)
    if seed % 2 == 0:
        pu.run_full_parity(w, strategy=strategy)


@pytest.mark.parametrize("seed", list(range(4)))
def test_staged_rows_equal_direct_on_large_random_layouts(oracle_lib, seed):
    w = big_random_workload(seed)
    R = 2
    a, b = run_rows(w, "direct", R), run_rows(w, "staged", R)
    for row in ("hsdp", "acc", "zero1"):
        if seed % 2 == 0:
            rows_vs_oracle(w, R, a, row)
        if row not in b:
            continue                  # the staged kernel does not hold this layout
        for x, y in zip(a[row], b[row]):
            if x is not None:
                assert torch.equal(_bits(x), _bits(y)), (row, w.N)
