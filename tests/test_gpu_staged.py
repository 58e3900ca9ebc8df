"""The two kernels behind fsdp_reduce_scatter_adamw (GPU).

direct: 16-byte loads straight into registers, one launch per alignment class.
staged: the bulk-copy engine stages each tile's state and gradient slices in
shared memory (mbarrier pipeline), one launch for both classes; beyond what two
stages hold (bf16 N > 16, fp32 N > 8) the replicas come in groups.

Each is compared with the oracle element by element on the same seeded inputs,
and the two with each other bit for bit.  The bounded-wait exit of the staged
pipeline is exercised with a wait that nothing completes: it must give up,
report FSDP_ETIMEOUT through fsdp_check_status, and leave the context usable.
"""
import numpy as np
import pytest
import torch

import fsdp_sharded_state_gb300 as fs
from fsdp_sharded_state_gb300 import synth

import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture
def rs_kernel():
    prev = fs.fsdp_set_rs_kernel("auto")
    yield fs.fsdp_set_rs_kernel
    fs.fsdp_set_rs_kernel(prev)


def W(shapes, units, N, mode, dtype, steps=2):
    return synth.Workload("staged_case", 9, list(shapes), list(units), N, mode, dtype, dtype, steps, 1e-3)


CASES = {
    "pad1": ([(5, 3), (4,)], [0, 0], 3, synth.FLAT),
    "odd_flat": ([(37, 5), (3,), (11, 13)], [0, 1, 1], 6, synth.FLAT),
    "odd_dim0": ([(37, 5), (3,), (11, 13)], [0, 0, 1], 6, synth.DIM0),
    "rowless": ([(1, 7)], [0], 5, synth.DIM0),
    "empty": ([(0, 4), (3,), (9, 0)], [0, 1, 1], 2, synth.DIM0),
    "scalar": ([(), (2,), (1000,)], [0, 0, 0], 3, synth.FLAT),
    "n1": ([(4099,)], [0], 1, synth.FLAT),
    "n16": ([(2049, 3), (17,)], [0, 0], 16, synth.FLAT),
    "n32": ([(5000, 3), (17,)], [0, 0], 32, synth.FLAT),         # replica groups
    "n64": ([(2049, 7), (9,)], [0, 0], 64, synth.FLAT),
    "n24_dim0": ([(700, 9), (33,), (50, 13)], [0, 0, 1], 24, synth.DIM0),
    "ragged": ([(1 << 16, 3)], [0], 7, synth.FLAT),
    "units": ([(300, 7), (5,), (64, 64), (33,)], [0, 1, 2, 2], 4, synth.FLAT),
}


@pytest.mark.parametrize("kind", ["direct", "staged"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("case", sorted(CASES))
def test_kernel_vs_oracle(oracle_lib, rs_kernel, kind, dtype, case):
    shapes, units, N, mode = CASES[case]
    rs_kernel(kind)
    pu.run_full_parity(W(shapes, units, N, mode, dtype))


@pytest.mark.parametrize("kind", ["direct", "staged"])
@pytest.mark.parametrize("P,N", [((1 << 20) + 1, 2), ((1 << 20) + 1, 8), (1 << 20, 16), ((1 << 20) + 3, 6),
                                 ((1 << 20) + 1, 32)])
def test_sweep_vs_oracle(oracle_lib, rs_kernel, kind, P, N):
    rs_kernel(kind)
    w = synth.sweep(P, N)
    w.steps = 2
    pu.run_full_parity(w)


@pytest.mark.parametrize("kind", ["direct", "staged"])
def test_reduced_llama_and_dim0_vs_oracle(oracle_lib, rs_kernel, kind):
    rs_kernel(kind)
    pu.run_full_parity(synth.llama4(blocks=1, hidden=256, ffn=688, N=8))
    pu.run_full_parity(synth.dim0_n6(vocab=320, hidden=64, ffn=176, N=6))
    pu.run_full_parity(synth.tiny_mlp())


def _run(w, kind, rs_kernel, steps=3):
    rs_kernel(kind)
    O = pu.oracle_offsets(w)
    st = pu.make_state(w, with_grad_out=True)
    st.init_from_full(synth.full_params(w, O["F"], O["t_full_off"], device="cuda"))
    for t in range(1, steps + 1):
        st.step(synth.grad_replicas(w, O["F"], t, device="cuda"), w.hp)
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("w", [
    synth.dim0_n6(vocab=3200, hidden=512, ffn=1376, N=6),                # many misaligned rank views
    W([(1 << 18, 3), (7,), (999, 5)], [0, 1, 1], 8, synth.FLAT, torch.float32),
    synth.sweep((1 << 22) + 1, 4),
    synth.sweep((1 << 21) + 1, 32),                                      # two replica groups
    W([(1 << 18, 3), (7,)], [0, 0], 32, synth.FLAT, torch.float32),      # three replica groups
], ids=["dim0_n6_small", "flat_f32_n8", "sweep_4M_n4", "sweep_2M_n32", "flat_f32_n32"])
def test_direct_and_staged_agree_bitwise(rs_kernel, w):
    a = _run(w, "direct", rs_kernel)
    b = _run(w, "staged", rs_kernel)
    for name in ("master", "exp_avg", "exp_avg_sq", "grad_out"):
        assert torch.equal(getattr(a, name).view(torch.int32), getattr(b, name).view(torch.int32)), name
    if a.param is not None:
        assert torch.equal(a.param.view(torch.int16), b.param.view(torch.int16))


def test_staged_refuses_what_does_not_fit(rs_kernel):
    rs_kernel("staged")
    with pytest.raises(fs.FsdpError):
        fs.fsdp_set_rs_kernel(7)
    # HSDP with 4 replica groups: more state copies than the staged kernel holds
    w = W([(4096,)], [0], 4, synth.FLAT, torch.bfloat16)
    L = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode)
    R, stride = 4, L.stride
    master = torch.zeros(R, w.N, stride, dtype=torch.float32, device="cuda")
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    grads = [torch.zeros(L.info["full_numel"], dtype=torch.bfloat16, device="cuda") for _ in range(R * w.N)]
    with pytest.raises(fs.FsdpError) as e:
        fs.fsdp_hsdp_reduce_scatter_adamw(L, 0, 1, R, grads, master, m, v, None, w.hp, 1)
    assert e.value.status == -1


def test_bounded_wait_gives_up_and_context_survives(oracle_lib, rs_kernel):
    fs.fsdp_check_status()
    fs.fsdp_wait_selftest(2_000_000)            # 2 ms
    with pytest.raises(fs.FsdpError) as e:
        fs.fsdp_check_status()
    assert e.value.status == -7                 # FSDP_ETIMEOUT
    fs.fsdp_check_status()                      # the record is cleared
    with pytest.raises(fs.FsdpError):
        fs.fsdp_wait_selftest(0)
    # the context is still usable: a staged step still matches the oracle
    rs_kernel("staged")
    pu.run_full_parity(synth.tiny_mlp())
    fs.fsdp_check_status()
