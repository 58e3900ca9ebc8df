"""The C-ABI library on the host (no GPU needed): it loads, exports every symbol
include/fsdp_state.h declares, computes layouts bit-exactly equal to the oracle's,
and rejects bad arguments with the documented status before launching anything.

Every rejected call below carries exactly one invalid argument, so validation
fails before any CUDA call; no call here can reach a kernel.
"""
import ctypes as C
import functools
import os
import re
import subprocess

import numpy as np
import pytest

import fsdp_sharded_state_gb300 as fs
import oracle
from fsdp_sharded_state_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fsdp_state.h")


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|void|size_t|const char\*)\s+(fsdp_\w+)\s*\(", src, re.M)))


def test_header_declares_the_binding_names():
    assert declared() == sorted(fs.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = fs.lib()
    for name in declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", fs.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (fsdp_\w+)$", out, re.M))
    assert set(declared()) <= exported


def seg_map(L, r):
    S = L.info["shard_numel"]
    m = np.full(S, -1, np.int64)
    for t in range(L.info["n_tensors"]):
        s = L.segment(t, r)
        m[s["shard_off"]:s["shard_off"] + s["len"]] = np.arange(s["full_off"], s["full_off"] + s["len"])
    return m


def small_cases():
    import random
    rng = random.Random(3)
    cases = [([(5, 3), (4,)], [0, 0], 3, 0), ([(5, 3)], [0], 4, 1), ([(1, 7)], [0], 5, 1),
             ([(0, 4), (3,)], [0, 1], 2, 1), ([(), (2,)], [0, 0], 2, 0), ([(2, 2), (3,), (1,)], [0, 1, 2], 4, 0)]
    for _ in range(120):
        T = rng.randint(1, 3)
        shapes = [tuple(rng.randint(0, 6) for _ in range(rng.randint(0, 3))) for _ in range(T)]
        units = [0]
        for _ in range(1, T):
            units.append(units[-1] + rng.randint(0, 1))
        cases.append((shapes, units, rng.randint(1, 9), rng.randint(0, 1)))
    return cases


@pytest.mark.parametrize("case", small_cases())
def test_layout_bit_exact_vs_oracle(oracle_lib, case):
    shapes, units, N, mode = case
    L = fs.Layout(shapes, units, N, mode)
    sh = oracle.Shapes(shapes, units)
    O = oracle.layout(sh, N, mode)
    info = L.info
    assert (info["numel"], info["shard_numel"], info["full_numel"], info["n_units"]) == (O["P"], O["S"], O["F"], O["U"])
    assert info["pad_numel"] == N * O["S"] - O["P"]
    assert info["shard_stride"] >= O["S"]
    assert info["shard_stride"] % 64 == 0 or info["shard_stride"] - O["S"] < 8
    for u in range(O["U"]):
        d = L.unit(u)
        assert (d["shard_off"], d["shard_numel"], d["full_off"], d["numel"]) == \
            (O["u_shard_off"][u], O["u_S"][u], O["u_full_off"][u], O["u_numel"][u])
    for t in range(len(shapes)):
        d = L.tensor(t)
        assert d["full_off"] == O["t_full_off"][t] and d["unit"] == units[t]
        if mode == 1:
            assert d["shard_off"] == O["t_shard_off"][t] and d["rows_per_rank"] == O["t_rows"][t]
    for r in range(N):
        exp = oracle.full_index(sh, N, mode, r, np.arange(O["S"]))
        assert np.array_equal(seg_map(L, r), exp)


@pytest.mark.parametrize("make", [synth.tiny_mlp, synth.mlp128m, synth.llama4, synth.dim0_n6,
                                  lambda: synth.sweep((1 << 29) + 1, 32), lambda: synth.sweep((1 << 20) + 1, 6)])
def test_workload_layouts_vs_oracle(oracle_lib, make):
    w = make()
    L = fs.Layout(w.shapes, w.unit_ids, w.N, w.mode)
    O = oracle.layout(oracle.Shapes(w.shapes, w.unit_ids), w.N, w.mode)
    assert (L.info["numel"], L.info["shard_numel"], L.info["full_numel"]) == (O["P"], O["S"], O["F"])
    for t in range(len(w.shapes)):
        assert L.tensor(t)["full_off"] == O["t_full_off"][t]
    # boundaries of every rank's view agree with the oracle's index map
    sh = oracle.Shapes(w.shapes, w.unit_ids)
    for t in range(len(w.shapes)):
        for r in range(w.N):
            s = L.segment(t, r)
            if s["len"] == 0:
                continue
            j = np.array([s["shard_off"], s["shard_off"] + s["len"] - 1])
            assert list(oracle.full_index(sh, w.N, w.mode, r, j)) == [s["full_off"], s["full_off"] + s["len"] - 1]


@pytest.mark.parametrize("case", small_cases()[:40])
@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_state_bytes_vs_oracle(oracle_lib, case, stage):
    shapes, units, N, mode = case
    L = fs.Layout(shapes, units, N, mode)
    sh = oracle.Shapes(shapes, units)
    for r in range(N):
        for phys in (True, False):
            assert L.state_bytes(stage, r, phys, 2, 4, 12, 4) == oracle.state_bytes(sh, N, mode, stage, r, phys,
                                                                                      2, 4, 12, 4)


@pytest.mark.parametrize("case", small_cases()[:40])
def test_collective_payload_vs_oracle(oracle_lib, case):
    shapes, units, N, mode = case
    L = fs.Layout(shapes, units, N, mode)
    sh = oracle.Shapes(shapes, units)
    keys = ("allreduce_input", "forward_allgather", "backward_allgather", "reducescatter_input", "broadcast")
    for strategy in range(5):
        for R in ((1, 2, 3) if strategy == fs.FSDP_HYBRID_SHARD else (1,)):
            got = L.collective_payload(strategy, R)
            elems, bus = oracle.collective_payload(sh, N, mode, strategy, R)
            assert [got[k] for k in keys] == elems, (strategy, R)
            assert got["bus_elements"] == pytest.approx(bus, rel=1e-12, abs=1e-9), (strategy, R)


def test_collective_payload_validation(lay):
    lib = fs.lib()
    out = fs.CollectivePayload()
    assert lib.fsdp_collective_payload(None, 3, 1, C.byref(out)) == -1
    assert lib.fsdp_collective_payload(lay.handle, 5, 1, C.byref(out)) == -1
    assert lib.fsdp_collective_payload(lay.handle, -1, 1, C.byref(out)) == -1
    assert lib.fsdp_collective_payload(lay.handle, 3, 2, C.byref(out)) == -1     # groups only with HSDP
    assert lib.fsdp_collective_payload(lay.handle, 4, 0, C.byref(out)) == -1
    assert lib.fsdp_collective_payload(lay.handle, 4, 2, None) == -1


# ---------------------------------------------------------------------------
# validation
# ---------------------------------------------------------------------------
def create_status(shapes, units, N, mode, dtypes=None):
    try:
        fs.Layout(shapes, units, N, mode, dtypes)
        return 0
    except fs.FsdpError as e:
        return e.status


def test_create_rejects_bad_descriptions():
    assert create_status([(4,)], [0], 0, 0) == -1                    # N < 1
    assert create_status([(4,)], [0], 65, 0) == -1                   # N > FSDP_MAX_RANKS
    assert create_status([(4,)], [0], 2, 7) == -1                    # unknown mode
    assert create_status([(4,), (4,)], [0, 2], 2, 0) == -3           # unit ids skip
    assert create_status([(4,)], [1], 2, 0) == -3                    # unit ids must start at 0
    assert create_status([(4, -1)], [0], 2, 0) == -3                 # negative dim
    assert create_status([(1 << 40, 1 << 40)], [0], 2, 0) == -5      # numel overflows int64
    assert create_status([(4,), (4,)], [0, 0], 2, 0, [0, 1]) == -2   # FlatParameter needs one dtype
    assert create_status([(4,), (4,)], [0, 1], 2, 0, [0, 1]) == 0    # ... per unit
    assert create_status([(4,), (4,)], [0, 0], 2, 1, [0, 1]) == 0    # DIM0 groups may mix
    assert create_status([(4,)], [0], 2, 0, [5]) == -2               # unknown dtype


@pytest.fixture
def lay():
    return fs.Layout([(64, 32), (64,)], [0, 1], 4, fs.FSDP_FLAT)


A = 1 << 20          # an aligned fake address: every call below fails before using it


def test_unshard_validation(lay):
    lib = fs.lib()
    assert lib.fsdp_unshard(None, 0, 1, A, A, 0, None) == -1
    assert lib.fsdp_unshard(lay.handle, 0, 3, A, A, 0, None) == -1      # unit range
    assert lib.fsdp_unshard(lay.handle, 1, 0, A, A, 0, None) == -1
    assert lib.fsdp_unshard(lay.handle, 0, 1, A, A, 9, None) == -2      # dtype
    assert lib.fsdp_unshard(lay.handle, 0, 1, None, A, 0, None) == -1   # NULL
    assert lib.fsdp_unshard(lay.handle, 0, 1, A + 4, A, 0, None) == -4  # misaligned
    assert lib.fsdp_unshard(lay.handle, 0, 1, A, A + 8, 0, None) == -4


def rs(lay, grads=None, gdt=1, master=A, m=A, v=A, param=None, gout=None, hp=(1e-3, 0.9, 0.999, 1e-8, 0.01),
       step=1, ub=0, ue=2, fn="fsdp_reduce_scatter_adamw"):
    lib = fs.lib()
    arr = (C.c_void_p * lay.N)(*(grads or [A] * lay.N))
    h = fs.AdamWHparams(*hp)
    return getattr(lib, fn)(lay.handle, ub, ue, arr, gdt, master, m, v, param, gout, C.byref(h), step, None)


# The allocating entry point and the one that allocates nothing make the same checks,
# all before any CUDA call: every rejection below runs on a machine with no GPU.
RS_ENTRY_POINTS = ["fsdp_reduce_scatter_adamw", "fsdp_reduce_scatter_adamw_noalloc"]


@pytest.mark.parametrize("fn", RS_ENTRY_POINTS)
def test_reduce_scatter_adamw_validation(lay, fn):
    rs = functools.partial(globals()["rs"], fn=fn)
    assert rs(lay, ue=3) == -1
    assert rs(lay, gdt=4) == -2
    assert rs(lay, step=0) == -1
    assert rs(lay, grads=[A, A, None, A]) == -1
    assert rs(lay, grads=[A, A, A + 2, A]) == -4
    assert rs(lay, master=None) == -1
    assert rs(lay, v=A + 4) == -4
    assert rs(lay, param=A + 2) == -4
    assert rs(lay, gout=A + 4) == -4
    for bad in [(-1e-3, .9, .999, 1e-8, .01), (1e-3, 1.0, .999, 1e-8, .01), (1e-3, .9, -0.1, 1e-8, .01),
                (1e-3, .9, .999, 0.0, .01), (1e-3, .9, .999, 1e-8, -1.0), (float("nan"), .9, .999, 1e-8, .01),
                (1e-3, .9, float("inf"), 1e-8, .01), (2.0, .9, .999, 1e-8, 0.6)]:
        assert rs(lay, hp=bad) == -1, bad
    assert rs(lay, ub=-1) == -1


def test_accumulate_reduce_scatter_adamw_validation(lay):
    lib = fs.lib()
    h = fs.AdamWHparams(1e-3, 0.9, 0.999, 1e-8, 0.01)

    def call(acc=None, micro=None, mdt=1, master=A, m=A, v=A, param=None, gout=None, hp=h, step=1, ub=0, ue=2,
             L=lay):
        a = (C.c_void_p * L.N)(*(acc or [A] * L.N))
        mi = (C.c_void_p * L.N)(*(micro or [A] * L.N))
        return lib.fsdp_accumulate_reduce_scatter_adamw(L.handle, ub, ue, a, mi, mdt, master, m, v, param, gout,
                                                        C.byref(hp), step, None)
    assert call(ue=3) == -1
    assert call(mdt=2) == -2
    assert call(step=0) == -1
    assert call(acc=[A, None, A, A]) == -1
    assert call(micro=[A, A, A + 2, A]) == -4
    assert call(acc=[A, A, A, A + 4]) == -4
    assert call(master=None) == -1
    assert call(v=A + 4) == -4
    assert call(param=A + 2) == -4
    assert call(gout=A + 8) == -4
    assert call(hp=fs.AdamWHparams(1e-3, 1.0, 0.999, 1e-8, 0.01)) == -1
    z = fs.Layout([(64, 32), (64,)], None, 4, fs.FSDP_ZERO1)
    assert call(L=z, ue=1) == -1


@pytest.mark.parametrize("fn", RS_ENTRY_POINTS)
def test_reduce_scatter_adamw_rejects_zero1_layouts(fn):
    # a ZeRO-1 layout keeps parameters whole: the reduce-scatter step does not apply
    z = fs.Layout([(64, 32), (64,)], None, 4, fs.FSDP_ZERO1)
    assert rs(z, fn=fn) == -1


def test_reshard_validation(lay):
    lib = fs.lib()
    assert lib.fsdp_reshard(lay.handle, 0, 2, None, 0, A, A, None) == 0      # release only: nothing launched
    assert lib.fsdp_reshard(lay.handle, 0, 5, None, 0, A, A, None) == -1
    assert lib.fsdp_reshard(lay.handle, 0, 2, A, 3, A, A, None) == -2
    assert lib.fsdp_reshard(lay.handle, 0, 2, A + 4, 0, A, A, None) == -4
    assert lib.fsdp_reshard(lay.handle, 0, 2, A, 0, None, None, None) == -1
    assert lib.fsdp_reshard(lay.handle, 0, 2, A, 0, A + 4, None, None) == -4


def test_queries_validation(lay):
    lib = fs.lib()
    x = C.c_int64()
    assert lib.fsdp_layout_unit(lay.handle, 2, None, None, None, None, None) == -1
    assert lib.fsdp_layout_tensor(lay.handle, -1, None, None, None, None, None) == -1
    assert lib.fsdp_layout_segment(lay.handle, 0, 4, C.byref(x), None, None, None) == -1
    out = (C.c_int64 * 3)()
    assert lib.fsdp_state_bytes(lay.handle, 4, 0, 1, 4, 4, 8, 0, out) == -1
    assert lib.fsdp_state_bytes(lay.handle, 3, 4, 1, 4, 4, 8, 0, out) == -1
    assert lib.fsdp_layout_query(None, None) == -1


def test_error_strings():
    for code, name in fs.STATUS.items():
        assert fs.fsdp_error_string(code).startswith(name)
    assert fs.fsdp_error_string(12345) == "unknown fsdp_status"


def test_kernel_choice_is_process_wide_and_checked():
    # the choice is host state: no GPU is touched
    prev = fs.fsdp_set_rs_kernel("direct")
    try:
        assert fs.fsdp_set_rs_kernel("staged") == fs.FSDP_RS_DIRECT
        assert fs.fsdp_set_rs_kernel("auto") == fs.FSDP_RS_STAGED
        for bad in (-1, 3, 99):
            assert fs.lib().fsdp_set_rs_kernel(bad) == -1          # FSDP_EINVAL, choice unchanged
        assert fs.fsdp_set_rs_kernel(fs.FSDP_RS_AUTO) == fs.FSDP_RS_AUTO
        with pytest.raises(KeyError):
            fs.fsdp_set_rs_kernel("fastest")
    finally:
        fs.fsdp_set_rs_kernel(prev)


def test_wait_selftest_validates_its_limit():
    for bad in (0, -5, 10_000_000_001):
        assert fs.lib().fsdp_wait_selftest(bad, None) == -1


@pytest.mark.parametrize("P", [(1 << 20) + 1, (1 << 24) + 3, (1 << 28) + 1, 4099, 1000003])
@pytest.mark.parametrize("N", [2, 3, 6, 8, 32])
def test_single_unit_flat_views_line_up(P, N):
    # One FLAT unit: the row stride is chosen so that every rank's view sits at a
    # shard index congruent to its full-layout index mod 8 (whole 16-byte vectors).
    L = fs.Layout([(P,)], [0], N, fs.FSDP_FLAT)
    for r in range(N):
        s = L.segment(0, r)
        if s["len"]:
            assert (s["full_off"] - (r * L.stride + s["shard_off"])) % 8 == 0, (P, N, r)


def test_rows_validation(lay):
    lib = fs.lib()
    h = fs.AdamWHparams(*synth.HP)
    g4 = (C.c_void_p * 4)(*([A] * 4))
    # clip: bad max_norm, missing workspace / grad shard, misaligned norm_out, ZeRO-1 layout
    clip = lambda **k: lib.fsdp_reduce_scatter_clip_adamw(
        k.get("L", lay.handle), 0, 2, g4, 1, A, A, A, None, k.get("gs", A), k.get("mx", 1.0), k.get("ws", A),
        k.get("no", None), C.byref(h), 1, None)
    assert clip(mx=0.0) == -1 and clip(mx=float("nan")) == -1 and clip(mx=-1.0) == -1
    assert clip(gs=None) == -1 and clip(ws=None) == -1 and clip(ws=A + 4) == -4 and clip(no=A + 4) == -4
    assert fs.fsdp_clip_workspace_bytes() >= 64 + 8 * 2 * 4096
    # accumulation: bad dtype, NULL / misaligned pointers
    acc = (C.c_void_p * 4)(*([A] * 4))
    assert lib.fsdp_accumulate_grads(lay.handle, 0, 2, acc, g4, 7, 1, None) == -2
    assert lib.fsdp_accumulate_grads(lay.handle, 0, 2, (C.c_void_p * 4)(A, A, None, A), g4, 1, 1, None) == -1
    assert lib.fsdp_accumulate_grads(lay.handle, 0, 2, acc, (C.c_void_p * 4)(A, A, A, A + 2), 1, 1, None) == -4
    assert lib.fsdp_accumulate_grads(lay.handle, 0, 3, acc, g4, 1, 1, None) == -1
    # HSDP: group count
    g8 = (C.c_void_p * 8)(*([A] * 8))
    assert lib.fsdp_hsdp_reduce_scatter_adamw(lay.handle, 0, 2, 0, g8, 1, A, A, A, None, C.byref(h), 1, None) == -1
    assert lib.fsdp_hsdp_reduce_scatter_adamw(lay.handle, 0, 2, 17, g8, 1, A, A, A, None, C.byref(h), 1,
                                              None) == -1   # 17 * 4 > 64 ranks
    # ZeRO-1 only on ZeRO-1 layouts; bf16 replicas need a master; fp32 replicas take none
    zl = fs.Layout([(7, 5), (3,), (9, 2)], None, 4, fs.FSDP_ZERO1)
    p4 = (C.c_void_p * 4)(*([A] * 4))
    z = lambda L, master, pdt: lib.fsdp_zero1_adamw_broadcast(L, 0, 1, g4, 1, master, A, A, p4, pdt, C.byref(h), 1,
                                                              None)
    assert z(lay.handle, None, 0) == -1
    assert z(zl.handle, None, 1) == -1 and z(zl.handle, A, 0) == -1
    # the other calls refuse ZeRO-1 layouts
    assert lib.fsdp_unshard(zl.handle, 0, 1, A, A, 0, None) == -1
    assert lib.fsdp_reduce_scatter_adamw(zl.handle, 0, 1, g4, 1, A, A, A, None, None, C.byref(h), 1, None) == -1
    owner = C.c_int32()
    assert lib.fsdp_layout_owner(lay.handle, 0, C.byref(owner)) == -1


def test_zero1_layout_vs_oracle_owners(oracle_lib):
    shapes = [(7, 5), (3,), (9, 2), (4, 4), (11,), (6, 6), (257, 33)]
    for N in (1, 2, 3, 4, 7):
        L = fs.Layout(shapes, None, N, fs.FSDP_ZERO1)
        owners = oracle.zero1_owners(oracle.Shapes(shapes), N)
        assert [L.owner(t) for t in range(len(shapes))] == list(owners)
        for t in range(len(shapes)):
            d = L.tensor(t)
            o = owners[t]
            assert (d["full_off"] - (o * L.stride + d["shard_off"])) % 8 == 0
            for r in range(N):
                s = L.segment(t, r)
                assert s["len"] == (int(np.prod(shapes[t])) if r == o else 0)
        # owner rows hold their tensors without overlap, inside the stride
        for r in range(N):
            spans = sorted((L.tensor(t)["shard_off"], L.tensor(t)["shard_off"] + int(np.prod(shapes[t])))
                           for t in range(len(shapes)) if owners[t] == r)
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 <= b0
            assert not spans or spans[-1][1] <= L.stride


# ---------------------------------------------------------------------------
# The step-constants block (host only)
def test_step_consts_block():
    import ctypes
    L = fs.Layout([(8, 3), (5,)], [0, 0], 6, fs.FSDP_FLAT)
    hp = (1e-3, 0.9, 0.999, 1e-8, 0.01)
    assert ctypes.sizeof(fs.AdamWStepConsts) == 48
    c1 = fs.fsdp_adamw_step_consts_make(L, hp, 1)
    assert c1.n_avg == 6.0
    assert c1.beta1 == np.float32(0.9) and c1.beta2 == np.float32(0.999) and c1.eps == np.float32(1e-8)
    b1, b2 = float(np.float32(0.9)), float(np.float32(0.999))
    lr, wd = float(np.float32(1e-3)), float(np.float32(0.01))
    # at step 1 the bias corrections are 1 - beta: step_size = lr / (1 - b1), bc2s = sqrt(1 - b2)
    assert c1.step_size == pytest.approx(lr / (1 - b1), rel=1e-6)
    assert c1.bc2s == pytest.approx((1 - b2) ** 0.5, rel=1e-6)
    assert c1.decay == pytest.approx(1 - lr * wd, rel=1e-7)
    assert c1.om1 == pytest.approx(1 - b1, rel=1e-6) and c1.om2 == pytest.approx(1 - b2, rel=1e-5)
    # late steps: the corrections go to 1
    c9 = fs.fsdp_adamw_step_consts_make(L, hp, 100000)
    assert c9.step_size == pytest.approx(lr, rel=1e-6) and c9.bc2s == pytest.approx(1.0, rel=1e-6)
    for bad_step, bad_hp in ((0, hp), (1, (1e-3, 1.0, 0.999, 1e-8, 0.01)), (1, (1e-3, 0.9, 0.999, 0.0, 0.01))):
        with pytest.raises(fs.FsdpError) as e:
            fs.fsdp_adamw_step_consts_make(L, bad_hp, bad_step)
        assert e.value.status == -1
