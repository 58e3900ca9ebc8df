"""Extreme inputs through the cast and the fused update (GPU), against the oracle.

Crafted bit patterns (synth.special_params / synth.special_grads) go through
fsdp_reshard, fsdp_unshard and fsdp_reduce_scatter_adamw:
  - parameters at exact bf16 round-to-nearest-even ties and next to them,
    subnormals, +-0, +-Inf, quiet and signalling NaNs, the largest finite values
    (which round up to Inf in bf16), large finite magnitudes;
  - gradients that are +-0 or subnormal in every replica, +-Inf or NaN in one
    replica, +Inf in one and -Inf in another, near the fp32 maximum in all (the sum
    overflows), of magnitude 1e19 .. 1e21 (the squared term (1-b2)*g*g overflows)
    or 1e-20 .. 1e-30 (it underflows);
  - eps down to the smallest subnormal, where the update of an element whose
    exp_avg_sq is 0 is exp_avg / eps.
The library is built without flush-to-zero, with IEEE division and square root
and no implicit contraction, and the oracle is plain C in binary32 with the same
operation order, so every result must agree bit for bit.  NaNs are compared by
position only: the pages fix no NaN payload, and the default NaN of a GPU
operation differs from a CPU's ("第18章 FSDP" §18.6 gives bf16 parameters cast from
the fp32 master; "NCCL ZeRO/FSDP state sharding", "ZeRO-2 方向", the reduce).

Layouts: both alignment classes (shard views congruent or not to their
full-layout position mod 8), DIM0 rows, fp32 replicas beyond one staging group
(N = 12) and bf16 replicas beyond one (N = 20); each test runs the automatic
kernel choice, the direct kernels and the staged kernels.
"""
import numpy as np
import pytest
import torch

import fsdp_sharded_state_gb300 as fs
import oracle
from fsdp_sharded_state_gb300 import synth

import parity_util as pu

pytestmark = pytest.mark.gpu

HP = synth.HP


def W(name, shapes, units, N, mode, dtype):
    return synth.Workload(name, 30, list(shapes), list(units), N, mode, dtype, dtype, 2, 1e-3)


LAYOUTS = [
    W("flat_bf16_n4", [(3000,), (1037, 3)], [0, 1], 4, synth.FLAT, torch.bfloat16),
    W("dim0_f32_n3", [(37, 65), (5,), (1500,)], [0, 0, 0], 3, synth.DIM0, torch.float32),
    W("flat_f32_n12", [(20000,)], [0], 12, synth.FLAT, torch.float32),
    W("flat_bf16_n20", [(5000,), (33,)], [0, 0], 20, synth.FLAT, torch.bfloat16),
]


@pytest.fixture(params=["auto", "direct", "staged"])
def kind(request):
    prev = fs.fsdp_set_rs_kernel(request.param)
    yield request.param
    fs.fsdp_set_rs_kernel(prev)


def is_nan_bf16(h):
    h = np.asarray(h, np.uint16)
    return ((h & 0x7F80) == 0x7F80) & ((h & 0x007F) != 0)


def assert_bits_f32(got, ref, what):
    """Bit for bit, NaNs by position."""
    got = np.ascontiguousarray(got, np.float32).reshape(-1)
    ref = np.ascontiguousarray(ref, np.float32).reshape(-1)
    gn, rn = np.isnan(got), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ ({gn.sum()} vs {rn.sum()})"
    bad = np.flatnonzero(got.view(np.uint32)[~rn] != ref.view(np.uint32)[~rn])
    if bad.size:
        i = np.flatnonzero(~rn)[bad[0]]
        raise AssertionError(f"{what}: {bad.size} elements differ, first at {i}: {got[i]!r} vs {ref[i]!r}")


def assert_bits_bf16(got, ref, what):
    got = np.ascontiguousarray(got, np.uint16).reshape(-1)
    ref = np.ascontiguousarray(ref, np.uint16).reshape(-1)
    gn, rn = is_nan_bf16(got), is_nan_bf16(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ"
    bad = np.flatnonzero(got[~rn] != ref[~rn])
    assert bad.size == 0, f"{what}: {bad.size} bf16 values differ, first {got[~rn][bad[0]]:#06x} vs {ref[~rn][bad[0]]:#06x}"


def to_dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32).view(np.int32)).cuda().view(torch.float32)


def to_dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def grads_for(w, F, seed):
    gd = "bf16" if w.grad_dtype == torch.bfloat16 else "f32"
    host = synth.special_grads(F, w.N, seed, gd)
    dev = [to_dev_bf16(g) if gd == "bf16" else to_dev_f32(g) for g in host]
    return host, dev


def start(w, full_np):
    """The CUDA state and the oracle state, both resharded from the same full buffer."""
    sh = oracle.Shapes(w.shapes, w.unit_ids)
    st = pu.make_state(w, with_grad_out=True)
    O = pu.oracle_offsets(w)
    assert st.F == O["F"]
    bf16 = w.param_dtype == torch.bfloat16
    st.init_from_full(to_dev_f32(full_np))
    om, op = oracle.reshard(sh, w.N, w.mode, full_np, st.stride, True, bf16)
    return sh, st, om, op


def compare(w, st, om, m, v, op, go, what):
    torch.cuda.synchronize()
    assert_bits_f32(pu.f32(st.master), om, f"master {what}")
    assert_bits_f32(pu.f32(st.exp_avg), m, f"exp_avg {what}")
    assert_bits_f32(pu.f32(st.exp_avg_sq), v, f"exp_avg_sq {what}")
    if go is not None:
        assert_bits_f32(pu.f32(st.grad_out), go, f"grad_out {what}")
    if op is not None:
        assert_bits_bf16(pu.u16(st.param), op, f"param {what}")


@pytest.mark.parametrize("w", LAYOUTS, ids=lambda w: w.name)
def test_reshard_and_unshard_of_special_values(oracle_lib, w):
    F = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode).info["full_numel"]
    full = synth.special_params(F, 11)
    sh, st, om, op = start(w, full)
    torch.cuda.synchronize()
    # the master is a copy of the full values: every bit, NaN payloads included
    assert np.array_equal(pu.f32(st.master).reshape(-1).view(np.uint32), om.view(np.uint32)), "reshard master"
    if op is not None:
        assert_bits_bf16(pu.u16(st.param), op, "reshard bf16 cast")
    st.unshard()
    ref = oracle.unshard(sh, w.N, w.mode, op if op is not None else om, st.stride, st.F)
    if op is not None:
        assert_bits_bf16(pu.u16(st.full), ref, "unshard")
    else:
        assert np.array_equal(pu.f32(st.full).view(np.uint32), ref.view(np.uint32)), "unshard"


@pytest.mark.parametrize("w", [LAYOUTS[0], LAYOUTS[3]], ids=lambda w: w.name)
def test_reshard_from_bf16_full_buffer(oracle_lib, w):
    """A bf16 full buffer widens exactly into the master and comes back unchanged."""
    sh = oracle.Shapes(w.shapes, w.unit_ids)
    st = pu.make_state(w)
    full16 = (synth.special_params(st.F, 12).view(np.uint32) >> 16).astype(np.uint16)
    fs.fsdp_reshard(st.layout, 0, st.layout.n_units, to_dev_bf16(full16), st.master, st.param)
    om, op = oracle.reshard(sh, w.N, w.mode, full16, st.stride, True, True)
    torch.cuda.synchronize()
    assert np.array_equal(pu.f32(st.master).reshape(-1).view(np.uint32), om.view(np.uint32)), "widened master"
    assert_bits_bf16(pu.u16(st.param), op, "param")


@pytest.mark.parametrize("w", LAYOUTS, ids=lambda w: w.name)
def test_cast_at_ties_through_the_update(oracle_lib, kind, w):
    """lr = 0, wd = 0: the update leaves every finite master value as it is, so the
    bf16 cast of the fused kernel meets the crafted ties, neighbours and overflows."""
    F = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode).info["full_numel"]
    full = synth.special_params(F, 13)
    sh, st, om, op = start(w, full)
    m, v, go = np.zeros_like(om), np.zeros_like(om), np.zeros_like(om)
    hp = (0.0, 0.9, 0.999, 1e-8, 0.0)
    for t in (1, 2):
        grads = synth.grad_replicas(w, F, t)
        st.reduce_scatter_adamw(grads, hp, step=t)
        oracle.rs_adamw(sh, w.N, w.mode, pu.grads_np(grads), st.stride, om, m, v, param=op, grad_out=go, hp=hp,
                        step=t)
        compare(w, st, om, m, v, op, go, f"step {t}")


@pytest.mark.parametrize("w", LAYOUTS, ids=lambda w: w.name)
def test_step_with_special_gradients(oracle_lib, kind, w):
    """Zero, subnormal, infinite, NaN, overflowing and underflowing gradients, two
    steps: the mean, the moments, the update and the cast, bit for bit."""
    F = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode).info["full_numel"]
    rng = np.random.default_rng(5)
    full = (rng.standard_normal(F) * 0.02).astype(np.float32)
    sh, st, om, op = start(w, full)
    m, v, go = np.zeros_like(om), np.zeros_like(om), np.zeros_like(om)
    for t in (1, 2):
        host, dev = grads_for(w, F, 100 + t)
        st.reduce_scatter_adamw(dev, HP, step=t)
        oracle.rs_adamw(sh, w.N, w.mode, host, st.stride, om, m, v, param=op, grad_out=go, hp=HP, step=t)
        compare(w, st, om, m, v, op, go, f"step {t}")
    # the crafted cases did occur: infinities and NaNs reached the state
    assert np.isinf(v).any() and np.isnan(om).any()


@pytest.mark.parametrize("eps", [1e-30, 1.17549435e-38, 1.4e-45])
@pytest.mark.parametrize("w", [LAYOUTS[0], LAYOUTS[2]], ids=lambda w: w.name)
def test_tiny_eps_with_zero_second_moment(oracle_lib, kind, w, eps):
    """eps down to the smallest subnormal: where exp_avg_sq is 0 (zero gradient, or a
    squared term that underflows) the update is exp_avg / eps, finite or not."""
    F = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode).info["full_numel"]
    rng = np.random.default_rng(7)
    full = (rng.standard_normal(F) * 0.02).astype(np.float32)
    sh, st, om, op = start(w, full)
    m, v, go = np.zeros_like(om), np.zeros_like(om), np.zeros_like(om)
    hp = (1e-3, 0.9, 0.999, eps, 0.01)
    for t in (1, 2):
        host, dev = grads_for(w, F, 200 + t)
        st.reduce_scatter_adamw(dev, hp, step=t)
        oracle.rs_adamw(sh, w.N, w.mode, host, st.stride, om, m, v, param=op, grad_out=go, hp=hp, step=t)
        compare(w, st, om, m, v, op, go, f"eps {eps} step {t}")
    assert ((v == 0) & (m != 0)).any()          # the case the test is for did occur
