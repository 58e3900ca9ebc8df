"""fsdp_reduce_scatter_adamw_noalloc against fsdp_reduce_scatter_adamw (GPU).

The no-allocation entry point serves callers that cannot call cudaMalloc (a
pre-sized pool or custom allocator that owns device memory, a step that must not
enter the driver's allocator, an embedder that forbids hidden allocations): its
segment table lives in a fixed array inside the library.  It must give the same
results as the allocating entry point, call after call, with either kernel.

This file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import fsdp_sharded_state_gb300 as fs
from fsdp_sharded_state_gb300 import synth

import parity_util as pu

pytestmark = pytest.mark.gpu


def _pair(w, with_grad_out):
    a = pu.make_state(w, with_grad_out=with_grad_out)
    b = pu.make_state(w, with_grad_out=with_grad_out)
    O = pu.oracle_offsets(w)
    full = synth.full_params(w, a.F, O["t_full_off"])
    a.init_from_full(full)
    b.init_from_full(full)
    return a, b


@pytest.mark.parametrize("w,ranges", [
    (synth.Workload("noalloc_dim0", 7, [(37, 5), (3,), (11, 13), (130, 64)], [0, 0, 1, 1], 6, synth.DIM0,
                    torch.bfloat16, torch.bfloat16, 2, 1e-3), [(0, 2)]),
    (synth.Workload("noalloc_flat", 7, [(300, 7), (5,), (64, 64), (33,)], [0, 1, 2, 2], 4, synth.FLAT,
                    torch.float32, torch.float32, 2, 1e-3), [(0, 1), (1, 3)]),
])
@pytest.mark.parametrize("with_grad_out", [False, True])
@pytest.mark.parametrize("kind", ["auto", "direct", "staged"])
def test_noalloc_matches_allocating_entry_point(w, ranges, with_grad_out, kind):
    prev = fs.fsdp_set_rs_kernel(kind)                 # both entry points follow the same choice
    try:
        _check_noalloc(w, ranges, with_grad_out)
    finally:
        fs.fsdp_set_rs_kernel(prev)


def _check_noalloc(w, ranges, with_grad_out):
    a, b = _pair(w, with_grad_out)
    lib = fs.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for t in (1, 2):                                   # two calls in a row
        grads = synth.grad_replicas(w, a.F, t)
        ptrs = (C.c_void_p * w.N)(*[g.data_ptr() for g in grads])
        h = fs.AdamWHparams(*w.hp)
        gdt = fs.FSDP_BF16 if w.grad_dtype == torch.bfloat16 else fs.FSDP_F32
        for ub, ue in ranges:
            a.reduce_scatter_adamw(grads, w.hp, step=t, ub=ub, ue=ue)
            rc = lib.fsdp_reduce_scatter_adamw_noalloc(
                b.layout.handle, ub, ue, ptrs, gdt, b.master.data_ptr(), b.exp_avg.data_ptr(),
                b.exp_avg_sq.data_ptr(), b.param.data_ptr() if b.param is not None else None,
                b.grad_out.data_ptr() if b.grad_out is not None else None, C.byref(h), t, stream)
            assert rc == 0, fs.fsdp_error_string(rc)
        fs.fsdp_check_status()
        for x, y, what in ((a.master, b.master, "master"), (a.exp_avg, b.exp_avg, "exp_avg"),
                           (a.exp_avg_sq, b.exp_avg_sq, "exp_avg_sq")):
            pu.assert_f32_close(pu.f32(y).reshape(-1), pu.f32(x).reshape(-1), f"{what} call {t}")
        if with_grad_out:
            pu.assert_f32_close(pu.f32(b.grad_out).reshape(-1), pu.f32(a.grad_out).reshape(-1), f"grad call {t}")
        if a.param is not None:
            pu.assert_bf16_close(pu.u16(b.param).reshape(-1), pu.u16(a.param).reshape(-1), f"param call {t}")


def test_noalloc_rejects_tables_beyond_its_scratch():
    # 200 tensors x 64 ranks = 12,800 pieces > FSDP_NOALLOC_MAX_SEGMENTS: refused, nothing launched.
    L = fs.Layout([(64, 8)] * 200, [0] * 200, 64, fs.FSDP_DIM0)
    A = 1 << 20                                        # never dereferenced: the size check fails first
    ptrs = (C.c_void_p * 64)(*([A] * 64))
    h = fs.AdamWHparams(*synth.HP)
    rc = fs.lib().fsdp_reduce_scatter_adamw_noalloc(L.handle, 0, 1, ptrs, fs.FSDP_BF16, A, A, A, A, None,
                                                    C.byref(h), 1, None)
    assert rc == -1


def test_noalloc_two_host_threads_on_one_stream():
    # Two host threads call the entry point at the same time on one stream, each for its
    # own layout and state.  Every call queues its table copy and its kernels together,
    # so each state ends as the allocating entry point leaves it, bit for bit.
    import threading
    wa = synth.Workload("noalloc_a", 7, [(300, 7), (5,), (64, 64)], [0, 1, 1], 4, synth.FLAT,
                        torch.bfloat16, torch.bfloat16, 2, 1e-3)
    wb = synth.Workload("noalloc_b", 8, [(37, 5), (3,), (130, 64)], [0, 0, 1], 6, synth.DIM0,
                        torch.float32, torch.float32, 2, 1e-3)
    K = 12
    side = torch.cuda.Stream()
    jobs = []
    for w in (wa, wb):
        ref, got = _pair(w, with_grad_out=True)
        grads = [synth.grad_replicas(w, ref.F, t) for t in range(1, K + 1)]
        for t in range(1, K + 1):
            ref.reduce_scatter_adamw(grads[t - 1], w.hp, step=t)
        jobs.append((w, ref, got, grads))
    torch.cuda.synchronize()
    lib = fs.lib()
    errors = []
    start = threading.Barrier(2)

    def worker(w, st, grads):
        try:
            h = fs.AdamWHparams(*w.hp)
            gdt = fs.FSDP_BF16 if w.grad_dtype == torch.bfloat16 else fs.FSDP_F32
            ptrs = [(C.c_void_p * w.N)(*[g.data_ptr() for g in gs]) for gs in grads]
            start.wait()
            for t in range(1, K + 1):
                rc = lib.fsdp_reduce_scatter_adamw_noalloc(
                    st.layout.handle, 0, st.layout.n_units, ptrs[t - 1], gdt, st.master.data_ptr(),
                    st.exp_avg.data_ptr(), st.exp_avg_sq.data_ptr(),
                    st.param.data_ptr() if st.param is not None else None, st.grad_out.data_ptr(), C.byref(h), t,
                    side.cuda_stream)
                assert rc == 0, fs.fsdp_error_string(rc)
        except BaseException as e:          # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(w, got, grads)) for w, _, got, grads in jobs]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    side.synchronize()
    fs.fsdp_check_status(side)
    assert not errors, errors
    for w, ref, got, _ in jobs:
        for name in ("master", "exp_avg", "exp_avg_sq", "grad_out", "param"):
            a, b = getattr(ref, name), getattr(got, name)
            if a is not None:
                assert torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                                   b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32)), (w.name, name)
