"""Edge cases of the CUDA path against the oracle (GPU).

Every buffer handed to the library is a real, large-enough device allocation;
no case here relies on the library catching an out-of-bounds or faulting access.
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


def W(shapes, units, N, mode, dtype=torch.bfloat16, steps=2, name="edge"):
    return synth.Workload(name, 9, list(shapes), list(units), N, mode, dtype, dtype, steps, 1e-3)


@pytest.mark.parametrize("case", [
    ([(5, 3), (4,)], [0, 0], 3, synth.FLAT),                    # one padding element
    ([(37, 5), (3,), (11, 13)], [0, 1, 1], 6, synth.FLAT),      # odd sizes: misaligned rank views
    ([(37, 5), (3,), (11, 13)], [0, 0, 1], 6, synth.DIM0),      # odd inner dims
    ([(1, 7)], [0], 5, synth.DIM0),                             # d0 < N: ranks own no row
    ([(0, 4), (3,), (9, 0)], [0, 1, 1], 2, synth.DIM0),         # empty tensors
    ([(), (2,), (1000,)], [0, 0, 0], 3, synth.FLAT),            # scalar
    ([(4099,)], [0], 1, synth.FLAT),                            # N = 1
    ([(2049, 3), (17,)], [0, 0], 64, synth.FLAT),               # N = 64 (the maximum)
    ([(130, 7)], [0], 64, synth.DIM0),
    ([(1 << 16, 3)], [0], 7, synth.FLAT),                       # many tiles, ragged tail
])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_edge_layouts(oracle_lib, case, dtype):
    shapes, units, N, mode = case
    pu.run_full_parity(W(shapes, units, N, mode, dtype))


def test_unit_ranges_touch_only_their_units(oracle_lib):
    w = W([(300, 7), (5,), (64, 64), (33,)], [0, 1, 2, 2], 4, synth.FLAT)
    st = pu.make_state(w)
    O = pu.oracle_offsets(w)
    full = synth.full_params(w, st.F, O["t_full_off"])
    st.init_from_full(full)
    before = [x.clone() for x in (st.master, st.exp_avg, st.exp_avg_sq, st.param)]
    grads = synth.grad_replicas(w, st.F, 1)
    st.reduce_scatter_adamw(grads, HP, step=1, ub=1, ue=2)
    st.reduce_scatter_adamw(grads, HP, step=1, ub=2, ue=2)     # empty range: nothing
    torch.cuda.synchronize()
    sh = oracle.Shapes(w.shapes, w.unit_ids)
    om, op = oracle.reshard(sh, w.N, w.mode, pu.f32(full), st.stride, True, True)
    m = np.zeros_like(om)
    v = np.zeros_like(om)
    oracle.rs_adamw(sh, w.N, w.mode, pu.grads_np(grads), st.stride, om, m, v, param=op, hp=HP, step=1, ub=1, ue=2)
    assert np.array_equal(pu.f32(st.master).reshape(-1).view(np.uint32), om.view(np.uint32))
    assert np.array_equal(pu.u16(st.param).reshape(-1), op)
    # units 0 and 2 untouched
    for u in (0, 2):
        a, n = O["u_shard_off"][u], O["u_S"][u]
        for x, x0 in zip((st.master, st.exp_avg, st.exp_avg_sq), before[:3]):
            assert torch.equal(x[:, a:a + n], x0[:, a:a + n])
    # unshard of unit 1 only writes unit 1's part of the full buffer
    sentinel = torch.full_like(st.full, 7.0)
    st.unshard(1, 2, out=sentinel)
    torch.cuda.synchronize()
    a, n = O["u_full_off"][1], w.N * O["u_S"][1]
    assert (sentinel[:a] == 7.0).all() and (sentinel[a + n:] == 7.0).all()
    ref = oracle.unshard(sh, w.N, w.mode, op, st.stride, st.F, ub=1, ue=2)
    assert np.array_equal(pu.u16(sentinel)[a:a + n], ref[a:a + n])


def test_grad_padding_is_never_read(oracle_lib):
    # FLAT padding positions of the gradient replicas hold NaN: no result may see it.
    w = W([(5, 3), (4,)], [0, 0], 3, synth.FLAT, torch.float32)
    st = pu.make_state(w, with_grad_out=True)
    O = pu.oracle_offsets(w)
    st.init_from_full(synth.full_params(w, st.F, O["t_full_off"]))
    grads = synth.grad_replicas(w, st.F, 1)
    for g in grads:
        g[O["P"]:] = float("nan")                    # the single padding slot at the end
    st.step(grads, HP)
    torch.cuda.synchronize()
    for x in (st.master, st.exp_avg, st.exp_avg_sq, st.grad_out):
        assert not torch.isnan(x).any()


def test_nan_propagates_to_its_element_only(oracle_lib):
    w = W([(64, 33)], [0], 4, synth.FLAT, torch.float32)
    st = pu.make_state(w)
    O = pu.oracle_offsets(w)
    st.init_from_full(synth.full_params(w, st.F, O["t_full_off"]))
    grads = synth.grad_replicas(w, st.F, 1)
    grads[2][100] = float("nan")
    st.step(grads, HP)
    torch.cuda.synchronize()
    sh = oracle.Shapes(w.shapes)
    nan = torch.isnan(st.master).reshape(-1).nonzero().reshape(-1).cpu().numpy()
    assert nan.size == 1
    r, j = divmod(int(nan[0]), st.stride)
    assert oracle.full_index(sh, w.N, w.mode, r, np.array([j]))[0] == 100


@pytest.mark.parametrize("mode", [synth.FLAT, synth.DIM0])
@pytest.mark.parametrize("full_dtype", [torch.float32, torch.bfloat16])
def test_reshard_unshard_round_trip(oracle_lib, mode, full_dtype):
    # summon_full_params(writeback): full -> shards -> full is the identity on logical
    # elements (bf16 shards of an fp32 full buffer are its rounding).
    w = W([(37, 5), (3,), (11, 13), (2,)], [0, 0, 1, 1], 6, mode)
    st = pu.make_state(w)
    O = pu.oracle_offsets(w)
    full = synth.full_params(w, st.F, O["t_full_off"], dtype=full_dtype)
    st.init_from_full(full)
    out = torch.zeros(st.F, dtype=torch.bfloat16, device="cuda")
    st.unshard(out=out)
    torch.cuda.synchronize()
    logical = np.zeros(st.F, bool)
    for t, s in enumerate(w.shapes):
        logical[O["t_full_off"][t]:O["t_full_off"][t] + int(np.prod(s))] = True
    exp = oracle.bf16_rne(pu.f32(full))
    assert np.array_equal(pu.u16(out)[logical], exp[logical])
    if mode == synth.FLAT:
        assert not pu.u16(out)[~logical].any()          # padding of the flat parameter is zero
    # fp32 master round trip
    st32 = fs.ShardedState(w.shapes, w.unit_ids, w.N, mode, param_dtype=torch.float32)
    st32.init_from_full(full)
    out32 = st32.unshard()
    torch.cuda.synchronize()
    assert np.array_equal(pu.f32(out32)[logical].view(np.uint32), pu.f32(full)[logical].view(np.uint32))


def test_canaries_around_buffers(oracle_lib):
    # The kernels write nothing outside the [N][stride] rows and the full buffer.
    w = W([(37, 5), (3,), (11, 13)], [0, 1, 1], 6, synth.FLAT)
    L = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode)
    N, stride, F = w.N, L.stride, L.info["full_numel"]
    pad = 1024
    CAN = 0x5A5A5A5A

    def arena(n, dtype):
        a = torch.empty(n + 2 * pad, dtype=dtype, device="cuda")
        a.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).fill_(0x5A5A if dtype == torch.bfloat16 else CAN)
        return a, a[pad:pad + n]

    arenas = {k: arena(N * stride, torch.float32) for k in ("master", "m", "v", "gout")}
    arenas["param"] = arena(N * stride, torch.bfloat16)
    arenas["full"] = arena(F, torch.bfloat16)
    O = pu.oracle_offsets(w)
    full32 = synth.full_params(w, F, O["t_full_off"])
    fs.fsdp_reshard(L, 0, L.n_units, full32, arenas["master"][1], arenas["param"][1])
    arenas["m"][1].zero_()
    arenas["v"][1].zero_()
    grads = synth.grad_replicas(w, F, 1)
    fs.fsdp_unshard(L, 0, L.n_units, arenas["param"][1], arenas["full"][1])
    fs.fsdp_reduce_scatter_adamw(L, 0, L.n_units, grads, arenas["master"][1], arenas["m"][1], arenas["v"][1],
                                 arenas["param"][1], arenas["gout"][1], HP, 1)
    fs.fsdp_check_status()
    for k, (a, _) in arenas.items():
        raw = a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32)
        c = 0x5A5A if a.dtype == torch.bfloat16 else CAN
        assert (raw[:pad] == c).all() and (raw[-pad:] == c).all(), k


def test_side_stream_and_two_layouts(oracle_lib):
    w1 = W([(300, 7)], [0], 4, synth.FLAT)
    w2 = W([(77, 9), (5,)], [0, 0], 3, synth.DIM0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = pu.make_state(w1)
        b = pu.make_state(w2)
        O1, O2 = pu.oracle_offsets(w1), pu.oracle_offsets(w2)
        a.init_from_full(synth.full_params(w1, a.F, O1["t_full_off"]))
        b.init_from_full(synth.full_params(w2, b.F, O2["t_full_off"]))
        ga, gb = synth.grad_replicas(w1, a.F, 1), synth.grad_replicas(w2, b.F, 1)
        a.step(ga, HP, stream=s)
        b.step(gb, HP, stream=s)
    fs.fsdp_check_status(s)
    for st, w, O, g in ((a, w1, O1, ga), (b, w2, O2, gb)):
        sh = oracle.Shapes(w.shapes, w.unit_ids)
        full = synth.full_params(w, st.F, O["t_full_off"])
        om, op = oracle.reshard(sh, w.N, w.mode, pu.f32(full), st.stride, True, True)
        m, v = np.zeros_like(om), np.zeros_like(om)
        oracle.rs_adamw(sh, w.N, w.mode, pu.grads_np(g), st.stride, om, m, v, param=op, hp=HP, step=1)
        assert np.array_equal(pu.f32(st.master).reshape(-1).view(np.uint32), om.view(np.uint32))
    a.layout.close()
    b.layout.close()
