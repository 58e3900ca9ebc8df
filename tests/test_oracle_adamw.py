"""Pins of the oracle's reduce-scatter + AdamW + bf16 cast (CPU).

Each pin checks the oracle against something other than itself:
  - the textbook AdamW (decoupled weight decay, bias-corrected moments, eps outside
    the root) evaluated in exact-ish fp64 for single elements over several steps;
  - the closed form of the first step (m = (1-b1) g, v = (1-b2) g^2, update ~ lr*sign(g));
  - torch.optim.AdamW (library routine) on the averaged gradient, within a band;
  - the pages' invariant that the sharded step equals the replicated (DDP) step;
  - the reduce = mean reading (sum over ranks, divided by N) and its fixed rank order,
    on hand-built values whose fp32 results are known exactly;
  - bf16 rounding against torch's float32 -> bfloat16 conversion.
"""
import numpy as np
import pytest
import torch

import oracle

HP = (1e-3, 0.9, 0.999, 1e-8, 0.01)


def f32(x):
    return np.float32(x)


def adamw_fp64(p, grads_per_step, lr, b1, b2, eps, wd):
    """Textbook AdamW in float64 (Loshchilov & Hutter with Kingma & Ba's bias correction)."""
    m = v = 0.0
    for t, g in enumerate(grads_per_step, start=1):
        p = p - lr * wd * p
        m = b1 * m + (1 - b1) * g
        v = b2 * v + (1 - b2) * g * g
        mhat = m / (1 - b1 ** t)
        vhat = v / (1 - b2 ** t)
        p = p - lr * mhat / (np.sqrt(vhat) + eps)
    return p, m, v


@pytest.mark.parametrize("seed", range(6))
def test_points_match_textbook_fp64(oracle_lib, seed):
    rng = np.random.default_rng(seed)
    n, N, steps = 64, 4, 5
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-3, (steps, n, N)).astype(np.float32)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(steps):
        oracle.adamw_points(g[t], p, m, v, want_param=False, hp=HP, step=t + 1)
    lr, b1, b2, eps, wd = (float(np.float32(x)) for x in HP)
    for i in range(n):
        gbar = [float(np.float64(g[t, i]).sum() / N) for t in range(steps)]
        pe, me, ve = adamw_fp64(float(p0[i]), gbar, lr, b1, b2, eps, wd)
        # fp32 vs fp64: a few roundings per step; m may cancel, so it gets an
        # absolute floor at 1e-6 of the gradient scale.
        assert abs(p[i] - pe) <= 2e-6 * abs(pe) + 1e-9
        assert abs(m[i] - me) <= 1e-5 * abs(me) + 1e-9
        assert abs(v[i] - ve) <= 1e-5 * abs(ve) + 1e-20


def test_first_step_closed_form(oracle_lib):
    # t = 1 from zero moments: m = (1-b1) g, v = (1-b2) g^2, bias-corrected update
    # lr * g / (|g| + eps), i.e. about lr * sign(g) when |g| >> eps.
    g = np.array([[3e-3], [-2e-2], [1e-5], [5.0]], np.float32)
    p0 = np.array([0.5, -0.25, 0.125, 1.0], np.float32)
    p, m, v = p0.copy(), np.zeros(4, np.float32), np.zeros(4, np.float32)
    oracle.adamw_points(g, p, m, v, want_param=False, hp=HP, step=1)
    lr, b1, b2, eps, wd = (float(np.float32(x)) for x in HP)     # the API's fp32 values
    gg = g[:, 0].astype(np.float64)
    assert np.allclose(m, (1 - b1) * gg, rtol=1e-6, atol=0)
    assert np.allclose(v, (1 - b2) * gg * gg, rtol=2e-6, atol=0)
    expect = p0 * (1 - lr * wd) - lr * gg / (np.abs(gg) + eps)
    assert np.allclose(p, expect, rtol=1e-6, atol=1e-9)
    assert abs((p0[3] * (1 - lr * wd) - p[3]) - lr) < 1e-7          # |g| >> eps: a step of lr


def test_reduce_is_mean_in_rank_order(oracle_lib):
    # N = 3: (1 + 2 + 4) / 3 rounded once.
    g = np.array([[1.0, 2.0, 4.0]], np.float32)
    p, m, v = np.zeros(1, np.float32), np.zeros(1, np.float32), np.zeros(1, np.float32)
    _, gout = oracle.adamw_points(g, p, m, v, want_param=False, want_grad=True, hp=HP, step=1)
    assert gout[0] == np.float32(7.0) / np.float32(3.0)
    # Rank order 0..N-1, left to right in fp32: ((1e8 + 1) - 1e8) + 1 = 1 (the first
    # +1 is absorbed), so the mean is 0.25 -- another order would give 0.5 or 0.
    g = np.array([[1e8, 1.0, -1e8, 1.0]], np.float32)
    _, gout = oracle.adamw_points(g, p, m, v, want_param=False, want_grad=True, hp=HP, step=1)
    assert gout[0] == np.float32(0.25)


def run_oracle_steps(shapes, units, N, mode, steps, seed, grad_bf16=False, param_bf16=True, ub=0, ue=None):
    sh = oracle.Shapes(shapes, units)
    L = oracle.layout(sh, N, mode)
    stride = L["S"] + 5                     # any stride >= S must give the same numbers
    rng = np.random.default_rng(seed)
    full = rng.normal(0, 0.02, L["F"]).astype(np.float32)
    master, param = oracle.reshard(sh, N, mode, full, stride, True, param_bf16)
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    gout = np.zeros_like(master)
    grads_all = []
    for t in range(1, steps + 1):
        g32 = [rng.normal(0, 1e-3, L["F"]).astype(np.float32) for _ in range(N)]
        grads = [oracle.bf16_rne(x) for x in g32] if grad_bf16 else g32
        grads_all.append(grads)
        oracle.rs_adamw(sh, N, mode, grads, stride, master, m, v, param=param, grad_out=gout, hp=HP, step=t,
                        ub=ub, ue=ue)
    return sh, L, stride, full, master, m, v, param, gout, grads_all


CASES = [
    ([(64, 32), (64,), (32, 64), (32,)], [0, 0, 0, 0], 4, oracle.FLAT),
    ([(5, 3), (4,)], [0, 0], 3, oracle.FLAT),
    ([(7, 5), (3,), (9, 2)], [0, 1, 1], 4, oracle.FLAT),
    ([(5, 3), (7,), (2, 4), (1, 6)], [0, 0, 1, 1], 3, oracle.DIM0),
    ([(13, 3), (4,)], [0, 0], 6, oracle.DIM0),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("grad_bf16", [False, True])
def test_sharded_equals_ddp_bitwise(oracle_lib, case, grad_bf16):
    """The sharded step, all-gathered, equals the replicated DDP step bit for bit
    ("NCCL ZeRO/FSDP state sharding", section 全模式性能结果与限制: all FSDP modes match
    ZeRO-0; "Optimizer Step 的所有权": the next all-gather recombines the shards)."""
    shapes, units, N, mode = case
    sh, L, stride, full0, master, m, v, param, gout, grads_all = run_oracle_steps(
        shapes, units, N, mode, steps=3, seed=11, grad_bf16=grad_bf16)
    # DDP: full fp32 state, the same averaged gradient, the same update.
    logical = np.zeros(L["F"], bool)
    for r in range(N):
        fi = oracle.full_index(sh, N, mode, r, np.arange(L["S"]))
        logical[fi[fi >= 0]] = True
    p = np.where(logical, full0, 0).astype(np.float32)
    pm = np.zeros_like(p)
    pv = np.zeros_like(p)
    for t, grads in enumerate(grads_all, start=1):
        oracle.ddp_adamw(grads, p, pm, pv, skip=~logical, hp=HP, step=t)
    got = oracle.unshard(sh, N, mode, master, stride, L["F"])
    assert np.array_equal(got[logical].view(np.uint32), p[logical].view(np.uint32))
    got_m = oracle.unshard(sh, N, mode, m, stride, L["F"])
    assert np.array_equal(got_m[logical].view(np.uint32), pm[logical].view(np.uint32))
    got_v = oracle.unshard(sh, N, mode, v, stride, L["F"])
    assert np.array_equal(got_v[logical].view(np.uint32), pv[logical].view(np.uint32))
    # bf16 copies are the rounding of the master
    assert np.array_equal(param, oracle.bf16_rne(master))


@pytest.mark.parametrize("case", CASES)
def test_padding_stays_positive_zero(oracle_lib, case):
    shapes, units, N, mode = case
    sh, L, stride, _, master, m, v, param, gout, _ = run_oracle_steps(shapes, units, N, mode, steps=3, seed=3)
    for r in range(N):
        fi = oracle.full_index(sh, N, mode, r, np.arange(L["S"]))
        pad = np.where(fi < 0)[0] + r * stride
        tail = np.arange(r * stride + L["S"], (r + 1) * stride)
        for arr in (master, m, v, gout):
            assert not arr[pad].view(np.uint32).any() and not arr[tail].view(np.uint32).any()
        assert not param[pad].any() and not param[tail].any()


def test_n1_is_plain_adamw(oracle_lib):
    shapes = [(6, 5), (4,)]
    sh, L, stride, full0, master, m, v, param, gout, grads_all = run_oracle_steps(
        shapes, [0, 0], 1, oracle.FLAT, steps=2, seed=5)
    assert L["S"] == L["P"] == L["F"]
    assert np.array_equal(oracle.full_index(sh, 1, oracle.FLAT, 0, np.arange(L["S"])), np.arange(L["S"]))
    p = full0.copy()
    pm = np.zeros_like(p)
    pv = np.zeros_like(p)
    for t, grads in enumerate(grads_all, start=1):
        oracle.adamw_points(grads[0][:, None], p, pm, pv, want_param=False, hp=HP, step=t)
    assert np.array_equal(master[:L["S"]].view(np.uint32), p.view(np.uint32))


def test_unit_range_touches_only_its_units(oracle_lib):
    shapes, units = [(7, 5), (3,), (9, 2)], [0, 1, 1]
    sh, L, stride, *_ = run_oracle_steps(shapes, units, 4, oracle.FLAT, steps=1, seed=9)
    sh, L, stride, full0, master, m, v, param, gout, _ = run_oracle_steps(
        shapes, units, 4, oracle.FLAT, steps=1, seed=9, ub=1, ue=2)
    master0, _ = oracle.reshard(sh, 4, oracle.FLAT, full0, stride, True, False)
    u0 = np.concatenate([np.arange(r * stride, r * stride + L["u_S"][0]) for r in range(4)])
    assert np.array_equal(master[u0], master0[u0])
    assert not m[u0].any()


def test_torch_adamw_band(oracle_lib):
    """torch.optim.AdamW on the averaged gradient agrees within a small band (the
    operation order differs, so not bit for bit)."""
    shapes, units, N = [(64, 32), (64,), (32, 64), (32,)], [0, 0, 0, 0], 4
    sh, L, stride, full0, master, m, v, param, gout, grads_all = run_oracle_steps(
        shapes, units, N, oracle.FLAT, steps=3, seed=21)
    w = torch.nn.Parameter(torch.from_numpy(full0.copy()))
    lr, b1, b2, eps, wd = (float(np.float32(x)) for x in HP)     # the API's fp32 values
    opt = torch.optim.AdamW([w], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd, foreach=False)
    for grads in grads_all:
        w.grad = torch.stack([torch.from_numpy(g) for g in grads]).double().mean(0).float()
        opt.step()
    got = oracle.unshard(sh, N, oracle.FLAT, master, stride, L["F"])
    ref = w.detach().numpy()
    # a few fp32 roundings apart: relative 1e-5, with an absolute floor of 1e-8
    # (ulp-level differences on values that crossed zero; the step size is 1e-3)
    err = np.abs(got - ref)
    assert (err <= 1e-5 * np.abs(ref) + 1e-8).all(), err.max()
    assert np.median(err / np.maximum(np.abs(ref), 1e-30)) < 1e-7
    st = opt.state[w]
    got_m = oracle.unshard(sh, N, oracle.FLAT, m, stride, L["F"])
    # torch forms m by lerp: ulp-of-g differences where m has cancelled
    assert np.allclose(got_m, st["exp_avg"].numpy(), rtol=1e-5, atol=1e-10)
    got_v = oracle.unshard(sh, N, oracle.FLAT, v, stride, L["F"])
    assert np.allclose(got_v, st["exp_avg_sq"].numpy(), rtol=1e-5, atol=1e-20)


def test_bf16_rne_matches_torch(oracle_lib):
    # Every sign/exponent/top-mantissa pattern, with low halves at and around the
    # rounding tie, plus a random sample; NaN compared as NaN.
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000], np.uint32)
    bits = (hi[:, None] | lows[None, :]).reshape(-1)
    rng = np.random.default_rng(0)
    bits = np.concatenate([bits, rng.integers(0, 1 << 32, 1 << 22, dtype=np.uint64).astype(np.uint32)])
    x = bits.view(np.float32)
    got = oracle.bf16_rne(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    g = got[nan]
    assert (((g & 0x7F80) == 0x7F80) & ((g & 0x007F) != 0)).all()       # still NaN
    assert np.array_equal(g >> 15, (bits[nan] >> 31).astype(np.uint16))  # sign kept
