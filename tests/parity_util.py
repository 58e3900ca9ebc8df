"""Helpers of the GPU parity tests: run the CUDA path and the oracle on the same
seeded inputs and compare.  The oracle gets its inputs from the seeded generators
(synth) and its layout from its own code, never from the CUDA path.

Tolerances (the stated bar): fp32 state (master, exp_avg, exp_avg_sq, reduced
gradient) max relative error <= 1e-6 (|x-ref| / max(|ref|, 1e-30)); bf16 params
<= 1 bf16 ulp; layout, unshard and reshard copies bit-exact.  With the same
reduction order and IEEE operations the expected difference is 0 ulp, and the
helpers report the ulp counts they saw.
"""
from __future__ import annotations

import numpy as np
import torch

import fsdp_sharded_state_gb300 as fs
import oracle
from fsdp_sharded_state_gb300 import synth

REL_TOL = 1e-6
BF16_ULP_TOL = 1


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().float().cpu().numpy()


def _ordered32(a):
    i = a.view(np.int32).astype(np.int64)
    return np.where(i < 0, -(i & 0x7FFFFFFF), i)


def _ordered16(a):
    i = a.astype(np.int64)
    return np.where(i & 0x8000, -(i & 0x7FFF), i)


def ulp_f32(a, b) -> int:
    if a.size == 0:
        return 0
    return int(np.abs(_ordered32(np.ascontiguousarray(a, np.float32)) -
                      _ordered32(np.ascontiguousarray(b, np.float32))).max())


def assert_f32_close(got, ref, what=""):
    got = np.ascontiguousarray(got, np.float32)
    ref = np.ascontiguousarray(ref, np.float32)
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN positions differ"
    g, r = got[~nan_r], ref[~nan_r]
    rel = np.abs(g.astype(np.float64) - r) / np.maximum(np.abs(r.astype(np.float64)), 1e-30)
    assert rel.size == 0 or rel.max() <= REL_TOL, f"{what}: max rel {rel.max():.3g}, max ulp {ulp_f32(g, r)}"
    return ulp_f32(g, r)


def assert_bf16_close(got_u16, ref_u16, what=""):
    got_u16 = np.ascontiguousarray(got_u16, np.uint16)
    ref_u16 = np.ascontiguousarray(ref_u16, np.uint16)
    if got_u16.size == 0:
        return 0
    d = np.abs(_ordered16(got_u16) - _ordered16(ref_u16)).max()
    assert d <= BF16_ULP_TOL, f"{what}: {d} bf16 ulp"
    return int(d)


def grads_np(grads):
    out = []
    for g in grads:
        out.append(u16(g) if g.dtype == torch.bfloat16 else f32(g))
    return out


def make_state(w: synth.Workload, device="cuda", with_grad_out=False):
    st = fs.ShardedState(w.shapes, w.unit_ids, w.N, w.mode, param_dtype=w.param_dtype, device=device,
                         with_grad_out=with_grad_out)
    return st


def oracle_offsets(w: synth.Workload):
    O = oracle.layout(oracle.Shapes(w.shapes, w.unit_ids), w.N, w.mode)
    return O


def run_full_parity(w: synth.Workload, steps=None, strategy="full_shard", with_grad_out=True, check_unshard=True):
    """Whole-state comparison after every step (small layouts)."""
    steps = w.steps if steps is None else steps
    sh = oracle.Shapes(w.shapes, w.unit_ids)
    O = oracle.layout(sh, w.N, w.mode)
    st = make_state(w, with_grad_out=with_grad_out)
    assert st.F == O["F"] and st.layout.info["shard_numel"] == O["S"]
    stride = st.stride
    full = synth.full_params(w, O["F"], O["t_full_off"], device="cuda")
    st.init_from_full(full)
    bf16 = w.param_dtype == torch.bfloat16
    om, op = oracle.reshard(sh, w.N, w.mode, f32(full), stride, True, bf16)
    assert np.array_equal(f32(st.master).reshape(-1).view(np.uint32), om.view(np.uint32)), "reshard master"
    if bf16:
        assert np.array_equal(u16(st.param).reshape(-1), op), "reshard bf16 param"
    m = np.zeros_like(om)
    v = np.zeros_like(om)
    go = np.zeros_like(om) if with_grad_out else None
    ulps = []
    for t in range(1, steps + 1):
        grads = synth.grad_replicas(w, O["F"], t, device="cuda")
        st.step(grads, w.hp, strategy=strategy)
        if check_unshard:
            # the all-gather of this step saw the parameters before the update
            ref_full = oracle.unshard(sh, w.N, w.mode, op if bf16 else om, stride, O["F"])
            got_full = u16(st.full) if bf16 else f32(st.full).view(np.uint32)
            refv = ref_full if bf16 else ref_full.view(np.uint32)
            assert np.array_equal(got_full, refv), f"unshard at step {t}"
        oracle.rs_adamw(sh, w.N, w.mode, grads_np(grads), stride, om, m, v, param=op if bf16 else None,
                        grad_out=go, hp=w.hp, step=t)
        torch.cuda.synchronize()
        u = [assert_f32_close(f32(st.master).reshape(-1), om, f"master step {t}"),
             assert_f32_close(f32(st.exp_avg).reshape(-1), m, f"exp_avg step {t}"),
             assert_f32_close(f32(st.exp_avg_sq).reshape(-1), v, f"exp_avg_sq step {t}")]
        if with_grad_out:
            u.append(assert_f32_close(f32(st.grad_out).reshape(-1), go, f"grad_out step {t}"))
        if bf16:
            u.append(assert_bf16_close(u16(st.param).reshape(-1), op, f"param step {t}"))
        ulps.append(max(u))
    return st, ulps


TILE = 2048          # elements of one kernel tile (256 threads x 8)


def sample_points(w: synth.Workload, O, n_random=200_000, seed=0, tile_frac=0.01):
    """(rank, j) sample of shard positions, with each one's full-layout index (-1 for
    padding, which is checked for +0): for every rank, the whole tile windows touching each
    boundary of every unit (FLAT) or tensor slot (DIM0) -- so every segment, rank and padding
    edge; a seeded random `tile_frac` of all tile windows, every element of each; and
    n_random seeded random positions."""
    sh = oracle.Shapes(w.shapes, w.unit_ids)
    rng = np.random.default_rng(seed)
    S = int(O["S"])
    bounds = set()
    if w.mode == oracle.FLAT:
        for u in range(O["U"]):
            a, n = int(O["u_shard_off"][u]), int(O["u_S"][u])
            own_last = int(O["u_numel"][u]) - (w.N - 1) * n           # logical elements of the last rank
            bounds.update((a, a + n, a + min(max(own_last, 0), n)))
    else:
        for t, shp in enumerate(w.shapes):
            a, n = int(O["t_shard_off"][t]), int(O["t_slot"][t])
            bounds.update((a, a + n))
            d0 = shp[0] if shp else 1
            inner = n // max(int(O["t_rows"][t]), 1) if n else 0
            for r in range(w.N):                                     # each rank's first padding row
                own = min(max(d0 - r * int(O["t_rows"][t]), 0), int(O["t_rows"][t]))
                bounds.add(a + own * inner)
    win = []
    for b in sorted(bounds):                                          # tiles touching a boundary
        lo = (max(b - 1, 0) // TILE) * TILE
        win.append(np.arange(lo, min(lo + 2 * TILE, S), dtype=np.int64))
    edge_j = np.unique(np.concatenate(win)) if win else np.zeros(0, np.int64)
    ranks, js = [], []
    for r in range(w.N):
        ranks.append(np.full(edge_j.size, r, np.int64))
        js.append(edge_j)
    n_tiles = (S + TILE - 1) // TILE
    k = max(1, int(round(tile_frac * w.N * n_tiles)))
    pick = rng.choice(w.N * n_tiles, size=min(k, w.N * n_tiles), replace=False)
    for p in pick:                                                     # whole random tiles
        r, t = divmod(int(p), n_tiles)
        j = np.arange(t * TILE, min((t + 1) * TILE, S), dtype=np.int64)
        ranks.append(np.full(j.size, r, np.int64))
        js.append(j)
    ranks.append(rng.integers(0, w.N, n_random))
    js.append(rng.integers(0, S, n_random))
    r = np.concatenate(ranks)
    j = np.concatenate(js)
    fi = np.empty_like(j)
    for q in range(w.N):
        sel = r == q
        fi[sel] = oracle.full_index(sh, w.N, w.mode, q, j[sel])
    return r.astype(np.int64), j, fi


def run_sampled_parity(w: synth.Workload, steps=None, strategy="full_shard", n_random=200_000,
                       with_grad_out=True):
    """Full-size run on the GPU, oracle on sampled points, tracked across steps.
    with_grad_out=False runs the kernel instance the bench times (no reduced-gradient
    output)."""
    steps = w.steps if steps is None else steps
    O = oracle_offsets(w)
    st = make_state(w, with_grad_out=with_grad_out)
    assert st.F == O["F"] and st.layout.info["shard_numel"] == O["S"]
    full = synth.full_params(w, O["F"], O["t_full_off"], device="cuda")
    st.init_from_full(full)
    r, j, fi = sample_points(w, O, n_random)
    lin = torch.from_numpy(r * st.stride + j).cuda()
    real = fi >= 0
    fi_t = torch.from_numpy(np.where(real, fi, 0)).cuda()
    p = np.where(real, f32(full[fi_t]), 0).astype(np.float32)      # the reshard: master = full value
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    bf16 = w.param_dtype == torch.bfloat16
    ulps = []
    for t in range(1, steps + 1):
        grads = synth.grad_replicas(w, O["F"], t, device="cuda")
        st.step(grads, w.hp, strategy=strategy)
        # the all-gather of this step: full[fi] == the pre-update bf16/fp32 parameter at (r, j)
        got_full = st.full[fi_t]
        if bf16:
            ref_par = oracle.bf16_rne(p)
            assert np.array_equal(u16(got_full)[real], ref_par[real]), f"unshard step {t}"
        else:
            assert np.array_equal(f32(got_full)[real].view(np.uint32), p[real].view(np.uint32)), f"unshard step {t}"
        g_rows = np.zeros((p.size, w.N), np.float32)
        for q in range(w.N):
            g_rows[:, q] = np.where(real, f32(grads[q][fi_t]), 0)
        par, gout = oracle.adamw_points(g_rows, p, m, v, want_param=True, want_grad=True, hp=w.hp, step=t)
        torch.cuda.synchronize()
        u = [assert_f32_close(f32(st.master.reshape(-1)[lin]), p, f"master step {t}"),
             assert_f32_close(f32(st.exp_avg.reshape(-1)[lin]), m, f"exp_avg step {t}"),
             assert_f32_close(f32(st.exp_avg_sq.reshape(-1)[lin]), v, f"exp_avg_sq step {t}")]
        if with_grad_out:
            u.append(assert_f32_close(f32(st.grad_out.reshape(-1)[lin]), gout, f"grad_out step {t}"))
        if bf16:
            u.append(assert_bf16_close(u16(st.param.reshape(-1)[lin]), par, f"param step {t}"))
        ulps.append(max(u))
        del grads
    # padding stays +0 (sampled padding positions went through the oracle with g = 0 too),
    # and so does every padding position of every state array, found from the oracle's layout
    pad = ~real
    assert not f32(st.master.reshape(-1)[lin])[pad].view(np.uint32).any()
    pads = torch.from_numpy(padding_positions(w, O, st.stride)).cuda()
    arrays = [("master", st.master), ("exp_avg", st.exp_avg), ("exp_avg_sq", st.exp_avg_sq), ("param", st.param),
              ("grad_out", st.grad_out)]
    for name, a in arrays:
        if a is not None and pads.numel():
            x = a.reshape(-1)[pads]
            assert not x.view(torch.int16 if x.dtype == torch.bfloat16 else torch.int32).any(), f"{name} padding"
    return st, ulps


def padding_positions(w: synth.Workload, O, stride):
    """Linear indices (rank * stride + j) of every padding element of the shard arrays,
    from the oracle's layout: FLAT -- the tail of each unit past its logical elements
    (on the last ranks); DIM0 -- each rank slot's rows past the rows it owns."""
    out = []
    for r in range(w.N):
        if w.mode == oracle.FLAT:
            for u in range(O["U"]):
                S_u, P_u, a = int(O["u_S"][u]), int(O["u_numel"][u]), int(O["u_shard_off"][u])
                own = min(max(P_u - r * S_u, 0), S_u)
                out.append(r * stride + np.arange(a + own, a + S_u, dtype=np.int64))
        else:
            for t, shp in enumerate(w.shapes):
                d0 = shp[0] if shp else 1
                inner = int(np.prod(shp[1:])) if len(shp) > 1 else 1
                c, a = int(O["t_rows"][t]), int(O["t_shard_off"][t])
                own = min(max(d0 - r * c, 0), c)
                out.append(r * stride + np.arange(a + own * inner, a + c * inner, dtype=np.int64))
    return np.concatenate(out) if out else np.zeros(0, np.int64)


def logical(O, shapes):
    """Mask of the full-layout positions that hold a tensor element (FLAT padding False)."""
    mask = np.zeros(O["F"], bool)
    for t, s in enumerate(shapes):
        mask[O["t_full_off"][t]:O["t_full_off"][t] + int(np.prod(s) if s else 1)] = True
    return mask


def oracle_zero1_rows(sh, N, owners):
    """The oracle's ZeRO-1 packing: each owner's tensors back to back, in tensor order;
    returns each tensor's offset in its owner's row and the row length."""
    sizes = [int(np.prod(s) if s else 1) for s in sh.shapes]
    off, fill = [], [0] * N
    for t, o in enumerate(owners):
        off.append(fill[o])
        fill[o] += sizes[t]
    return off, max(fill)
