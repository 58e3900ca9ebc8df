"""The fused step with its AdamW constants in device memory, and the step captured in
CUDA graphs (GPU).

fsdp_reduce_scatter_adamw_consts must give fsdp_reduce_scatter_adamw's results bit for
bit when its device block holds the same step's constants; StepGraph (the step
captured once, replayed with the constants rewritten before each replay) must give
the eager step's results bit for bit, step after step."""
import ctypes

import numpy as np
import pytest
import torch

import fsdp_sharded_state_gb300 as fs
from fsdp_sharded_state_gb300 import synth

import parity_util as pu

pytestmark = pytest.mark.gpu


def W(shapes, units, N, mode, dtype=torch.bfloat16, steps=3):
    return synth.Workload("graph", 13, list(shapes), list(units), N, mode, dtype, dtype, steps, 1e-3)


CASES = [W([(300, 37), (13,), (64, 65)], [0, 0, 1], 4, synth.FLAT),
         W([(130, 64), (7,), (9, 3)], [0, 0, 0], 6, synth.DIM0),
         W([(512, 96), (96,)], [0, 0], 4, synth.FLAT, torch.float32),
         W([((1 << 16) + 1,)], [0], 32, synth.FLAT)]                      # replica groups


def _same(a, b, what):
    if a is None and b is None:
        return
    ia = a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16)
    ib = b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16)
    assert torch.equal(ia, ib), what


def _pair(w, with_grad_out):
    a, b = pu.make_state(w, with_grad_out=with_grad_out), pu.make_state(w, with_grad_out=with_grad_out)
    O = pu.oracle_offsets(w)
    full = synth.full_params(w, a.F, O["t_full_off"])
    a.init_from_full(full)
    b.init_from_full(full)
    return a, b


@pytest.mark.parametrize("block", ["device", "pinned_host"])
@pytest.mark.parametrize("with_grad_out", [False, True])
@pytest.mark.parametrize("w", CASES)
def test_consts_call_equals_fused_call(oracle_lib, w, with_grad_out, block):
    """The block in device memory (uploaded on the stream) or read by the kernel from
    page-locked host memory."""
    a, b = _pair(w, with_grad_out)
    L = b.layout
    dev = torch.zeros(12, dtype=torch.float32, device="cuda")
    host = torch.zeros(12, dtype=torch.float32).pin_memory()
    for t in (1, 2, 3):
        grads = [g.to(w.grad_dtype) for g in synth.grad_replicas(w, a.F, t)]
        a.reduce_scatter_adamw(grads, w.hp, step=t)
        c = fs.fsdp_adamw_step_consts_make(L, w.hp, t)
        torch.cuda.synchronize()                      # host block free to rewrite
        ctypes.memmove(host.data_ptr(), ctypes.addressof(c), 48)
        if block == "device":
            fs.fsdp_adamw_step_consts_upload(dev, host)
        fs.fsdp_reduce_scatter_adamw_consts(L, 0, L.n_units, grads, b.master, b.exp_avg, b.exp_avg_sq, b.param,
                                            b.grad_out, consts=dev if block == "device" else host)
        torch.cuda.synchronize()
        for x, y, what in ((a.master, b.master, "master"), (a.exp_avg, b.exp_avg, "exp_avg"),
                           (a.exp_avg_sq, b.exp_avg_sq, "exp_avg_sq"), (a.param, b.param, "param"),
                           (a.grad_out, b.grad_out, "grad_out")):
            _same(x, y, f"{what} step {t}")


@pytest.mark.parametrize("with_grad_out", [False, True])
@pytest.mark.parametrize("strategy", ["full_shard", "shard_grad_op"])
@pytest.mark.parametrize("w", [synth.tiny_mlp()] + CASES[:3])
def test_step_graph_equals_eager(oracle_lib, w, strategy, with_grad_out):
    """Six steps: the first runs eagerly and captures the graphs, five replay them
    (the three host blocks each come round twice).  With the reduced-gradient output,
    the graphs also hold the zero-fill of its padding."""
    a, b = _pair(w, with_grad_out)
    grads = [g.to(w.grad_dtype) for g in synth.grad_replicas(w, a.F, 1)]
    g = fs.StepGraph(b, grads, w.hp, strategy, n_blocks=3)
    for t in range(1, 7):
        a.step(grads, w.hp, strategy=strategy)
        g.step()
        torch.cuda.synchronize()
        assert a.t == b.t == t
        for x, y, what in ((a.master, b.master, "master"), (a.exp_avg, b.exp_avg, "exp_avg"),
                           (a.exp_avg_sq, b.exp_avg_sq, "exp_avg_sq"), (a.param, b.param, "param"),
                           (a.full, b.full, "gathered buffer"), (a.grad_out, b.grad_out, "grad_out")):
            _same(x, y, f"{what} step {t}")
    fs.fsdp_check_status()


def test_step_graph_refilled_gradients(oracle_lib):
    """The graph reads the gradient buffers it was captured with: refilling them in
    place between replays gives the eager steps on the new values."""
    w = synth.tiny_mlp()
    a, b = _pair(w, False)
    grads = [torch.empty(a.F, dtype=w.grad_dtype, device="cuda") for _ in range(w.N)]
    g = fs.StepGraph(b, grads, w.hp)
    for t in range(1, 5):
        for q, x in enumerate(synth.grad_replicas(w, a.F, t)):
            grads[q].copy_(x.to(w.grad_dtype))
        a.step(grads, w.hp)
        g.step()
    torch.cuda.synchronize()
    _same(a.master, b.master, "master")
    _same(a.exp_avg_sq, b.exp_avg_sq, "exp_avg_sq")
    _same(a.full, b.full, "gathered buffer")


def test_consts_rejects_bad_arguments(oracle_lib):
    w = CASES[0]
    st = pu.make_state(w)
    L = st.layout
    grads = [g.to(w.grad_dtype) for g in synth.grad_replicas(w, st.F, 1)]
    dev = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(fs.FsdpError) as e:                          # misaligned block
        fs.fsdp_reduce_scatter_adamw_consts(L, 0, L.n_units, grads, st.master, st.exp_avg, st.exp_avg_sq,
                                            st.param, None, consts=dev[1:])
    assert e.value.status == -4
    with pytest.raises(fs.FsdpError) as e:                          # no block
        fs.fsdp_reduce_scatter_adamw_consts(L, 0, L.n_units, grads, st.master, st.exp_avg, st.exp_avg_sq,
                                            st.param, None, consts=None)
    assert e.value.status == -1
    with pytest.raises(fs.FsdpError) as e:                          # no host source
        fs.fsdp_adamw_step_consts_upload(dev, None)
    assert e.value.status == -1
    pageable = np.zeros(16, np.float32)                             # not page-locked: refused
    addr = pageable.ctypes.data
    addr += (-addr) % 16
    with pytest.raises(fs.FsdpError) as e:
        fs.fsdp_reduce_scatter_adamw_consts(L, 0, L.n_units, grads, st.master, st.exp_avg, st.exp_avg_sq,
                                            st.param, None, consts=addr)
    assert e.value.status == -1
    torch.cuda.synchronize()
    assert not np.any(pu.f32(st.exp_avg))                           # nothing was launched
