"""Python loader for the plain-C oracle of the sharded-state step.

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` import this package.  The product path never does.

The C source (``oracle.c``) restates what the FSDP pages compute: the
FlatParameter / dim-0 layout, the all-gather, the mean reduce-scatter in fp32,
AdamW on the fp32 shard and the bf16 recast.  This module only marshals numpy
arrays into it; it holds none of the arithmetic.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "_build", "liboracle.so")

FLAT, DIM0 = 0, 1
F32, BF16 = 0, 1

# Compiler flags: IEEE binary32 arithmetic, no implicit contraction, no fast-math.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc)."""
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"])
        os.replace(tmp, LIB)
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _lib.oracle_bf16_rne.restype = C.c_uint16
        _lib.oracle_bf16_rne.argtypes = [C.c_float]
    return _lib


def _p(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


class Shapes:
    """A tensor list: shapes plus the unit (wrap unit / param group) of each."""

    def __init__(self, shapes, unit_ids=None):
        self.shapes = [tuple(int(d) for d in s) for s in shapes]
        self.T = len(self.shapes)
        self.ndim = np.array([len(s) for s in self.shapes], dtype=np.int32)
        self.dims = np.array([d for s in self.shapes for d in s] or [0], dtype=np.int64)
        if unit_ids is None:
            unit_ids = [0] * self.T
        self.unit = np.array(unit_ids, dtype=np.int32)

    def args(self):
        return (C.c_int32(self.T), _p(self.ndim), _p(self.dims), _p(self.unit))


def layout(sh: Shapes, N: int, mode: int) -> dict:
    T = sh.T
    scal = np.zeros(5, np.int64)
    arrs = {k: np.zeros(T, np.int64) for k in
            ("t_full_off", "t_shard_off", "t_rows", "t_slot", "u_S", "u_shard_off", "u_full_off", "u_numel")}
    rc = lib().oracle_layout(*sh.args(), C.c_int32(N), C.c_int32(mode), _p(scal),
                             *[_p(arrs[k]) for k in ("t_full_off", "t_shard_off", "t_rows", "t_slot",
                                                     "u_S", "u_shard_off", "u_full_off", "u_numel")])
    if rc != 0:
        raise ValueError("oracle_layout rejected the description")
    P, S, F, U, _ = (int(x) for x in scal)
    out = {"P": P, "S": S, "F": F, "U": U, "N": N, "mode": mode}
    for k, v in arrs.items():
        out[k] = v[:U].copy() if k.startswith("u_") else v.copy()
    return out


def full_index(sh: Shapes, N: int, mode: int, rank: int, j) -> np.ndarray:
    j = np.ascontiguousarray(j, dtype=np.int64)
    out = np.empty_like(j)
    rc = lib().oracle_full_index(*sh.args(), C.c_int32(N), C.c_int32(mode), C.c_int32(rank),
                                 C.c_int64(j.size), _p(j), _p(out))
    if rc != 0:
        raise ValueError("oracle_full_index failed")
    return out


def reshard(sh, N, mode, full, stride, want_master=True, want_param=True):
    full = np.ascontiguousarray(full)
    fdt = BF16 if full.dtype == np.uint16 else F32
    master = np.empty(N * stride, np.float32) if want_master else None
    param = np.empty(N * stride, np.uint16) if want_param else None
    rc = lib().oracle_reshard(*sh.args(), C.c_int32(N), C.c_int32(mode), _p(full), C.c_int32(fdt),
                              C.c_int64(stride), _p(master), _p(param))
    if rc != 0:
        raise ValueError("oracle_reshard failed")
    return master, param


def unshard(sh, N, mode, shards, stride, F, ub=0, ue=None, out=None):
    shards = np.ascontiguousarray(shards)
    if ue is None:
        ue = int(sh.unit[-1]) + 1
    if out is None:
        out = np.zeros(F, shards.dtype)
    rc = lib().oracle_unshard(*sh.args(), C.c_int32(N), C.c_int32(mode), C.c_int32(ub), C.c_int32(ue),
                              _p(shards), C.c_int32(shards.dtype.itemsize), C.c_int64(stride), _p(out))
    if rc != 0:
        raise ValueError("oracle_unshard failed")
    return out


def _grad_ptrs(grads):
    grads = [np.ascontiguousarray(g) for g in grads]
    dt = BF16 if grads[0].dtype == np.uint16 else F32
    arr = (C.c_void_p * len(grads))(*[g.ctypes.data for g in grads])
    return grads, arr, dt


def rs_adamw(sh, N, mode, grads, stride, master, m, v, param=None, grad_out=None,
             hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step=1, ub=0, ue=None):
    """In place on master/m/v (and param/grad_out when given)."""
    if ue is None:
        ue = int(sh.unit[-1]) + 1
    keep, arr, dt = _grad_ptrs(grads)
    lr, b1, b2, eps, wd = hp
    rc = lib().oracle_rs_adamw(*sh.args(), C.c_int32(N), C.c_int32(mode), C.c_int32(ub), C.c_int32(ue),
                               arr, C.c_int32(dt), C.c_int64(stride), _p(master), _p(m), _p(v),
                               _p(param), _p(grad_out), C.c_float(lr), C.c_float(b1), C.c_float(b2),
                               C.c_float(eps), C.c_float(wd), C.c_int64(step))
    if rc != 0:
        raise ValueError("oracle_rs_adamw failed")


def ddp_adamw(grads, p, m, v, skip=None, hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step=1):
    keep, arr, dt = _grad_ptrs(grads)
    lr, b1, b2, eps, wd = hp
    skip_a = None if skip is None else np.ascontiguousarray(skip, dtype=np.uint8)
    rc = lib().oracle_ddp_adamw(C.c_int64(p.size), C.c_int32(len(keep)), arr, C.c_int32(dt), _p(skip_a),
                                _p(p), _p(m), _p(v), C.c_float(lr), C.c_float(b1), C.c_float(b2),
                                C.c_float(eps), C.c_float(wd), C.c_int64(step))
    if rc != 0:
        raise ValueError("oracle_ddp_adamw failed")


def adamw_points(g_rows, p, m, v, want_param=True, want_grad=False,
                 hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step=1):
    """g_rows: [n, N] fp32 replica gradients per point.  In place on p/m/v."""
    g_rows = np.ascontiguousarray(g_rows, dtype=np.float32)
    n, N = g_rows.shape
    param = np.empty(n, np.uint16) if want_param else None
    gout = np.empty(n, np.float32) if want_grad else None
    lr, b1, b2, eps, wd = hp
    rc = lib().oracle_adamw_points(C.c_int64(n), C.c_int32(N), _p(g_rows), _p(p), _p(m), _p(v),
                                   _p(param), _p(gout), C.c_float(lr), C.c_float(b1), C.c_float(b2),
                                   C.c_float(eps), C.c_float(wd), C.c_int64(step))
    if rc != 0:
        raise ValueError("oracle_adamw_points failed")
    return param, gout


def bf16_rne(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_bf16_rne_array(C.c_int64(x.size), _p(x), _p(out))
    return out


def state_bytes(sh, N, mode, stage, rank, physical, pb, gb, ob, step_bytes=0):
    out = np.zeros(3, np.int64)
    rc = lib().oracle_state_bytes(*sh.args(), C.c_int32(N), C.c_int32(mode), C.c_int32(stage),
                                  C.c_int32(rank), C.c_int32(int(physical)), C.c_int64(pb), C.c_int64(gb),
                                  C.c_int64(ob), C.c_int64(step_bytes), _p(out))
    if rc != 0:
        raise ValueError("oracle_state_bytes failed")
    return tuple(int(x) for x in out)


NO_SHARD, ZERO1_OPT, SHARD_GRAD_OP, FULL_SHARD, HYBRID_SHARD = 0, 1, 2, 3, 4


def collective_payload(sh, N, mode, strategy, R=1):
    """Per-rank collective payload of one step: (elems, bus) with elems = all-reduce
    input, forward all-gather, backward all-gather, reduce-scatter input, broadcast
    (logical elements) and bus = elements a rank sends under ring algorithms."""
    elems = np.zeros(5, np.int64)
    bus = C.c_double()
    rc = lib().oracle_collective_payload(*sh.args(), C.c_int32(N), C.c_int32(mode), C.c_int32(strategy),
                                         C.c_int32(R), _p(elems), C.byref(bus))
    if rc != 0:
        raise ValueError("oracle_collective_payload rejected the arguments")
    return [int(x) for x in elems], bus.value


def rs_clip_adamw(sh, N, mode, grads, stride, master, m, v, max_norm, param=None, grad_out=None,
                  hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step=1, ub=0, ue=None):
    """Reduce-scatter, sharded clip_grad_norm_, AdamW; in place.  Returns the norm."""
    if ue is None:
        ue = int(sh.unit[-1]) + 1
    keep, arr, dt = _grad_ptrs(grads)
    lr, b1, b2, eps, wd = hp
    norm = C.c_double()
    rc = lib().oracle_rs_clip_adamw(*sh.args(), C.c_int32(N), C.c_int32(mode), C.c_int32(ub), C.c_int32(ue),
                                    arr, C.c_int32(dt), C.c_int64(stride), _p(master), _p(m), _p(v), _p(param),
                                    _p(grad_out), C.c_float(max_norm), C.c_float(lr), C.c_float(b1), C.c_float(b2),
                                    C.c_float(eps), C.c_float(wd), C.c_int64(step), C.byref(norm))
    if rc != 0:
        raise ValueError("oracle_rs_clip_adamw failed")
    return norm.value


def accumulate(acc, micro, first):
    """acc = micro (first) or acc + micro, fp32, in place."""
    micro = np.ascontiguousarray(micro)
    dt = BF16 if micro.dtype == np.uint16 else F32
    rc = lib().oracle_accumulate(C.c_int64(acc.size), _p(acc), _p(micro), C.c_int32(dt), C.c_int32(int(first)))
    if rc != 0:
        raise ValueError("oracle_accumulate failed")


def hsdp_adamw(sh, N, mode, R, grads, stride, master, m, v, param=None, hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step=1):
    """grads: R*N replicas (group-major).  master/m/v/param: R copies of [N][stride]."""
    keep, arr, dt = _grad_ptrs(grads)
    lr, b1, b2, eps, wd = hp
    rc = lib().oracle_hsdp_adamw(*sh.args(), C.c_int32(N), C.c_int32(mode), C.c_int32(R), arr, C.c_int32(dt),
                                 C.c_int64(stride), _p(master), _p(m), _p(v), _p(param), C.c_float(lr),
                                 C.c_float(b1), C.c_float(b2), C.c_float(eps), C.c_float(wd), C.c_int64(step))
    if rc != 0:
        raise ValueError("oracle_hsdp_adamw failed")


def zero1_owners(sh, N):
    owner = np.zeros(sh.T, np.int32)
    rc = lib().oracle_zero1_owners(C.c_int32(sh.T), _p(sh.ndim), _p(sh.dims), C.c_int32(N), _p(owner))
    if rc != 0:
        raise ValueError("oracle_zero1_owners failed")
    return owner


def zero1_adamw(sh, N, grads, stride, master, m, v, params, hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step=1):
    """params: N full replicas (fp32, or uint16 bf16 when master is given); in place."""
    keep, arr, dt = _grad_ptrs(grads)
    params = [np.ascontiguousarray(p) for p in params]
    parr = (C.c_void_p * N)(*[p.ctypes.data for p in params])
    lr, b1, b2, eps, wd = hp
    rc = lib().oracle_zero1_adamw(C.c_int32(sh.T), _p(sh.ndim), _p(sh.dims), C.c_int32(N), arr, C.c_int32(dt),
                                  C.c_int64(stride), _p(master), _p(m), _p(v), parr, C.c_float(lr), C.c_float(b1),
                                  C.c_float(b2), C.c_float(eps), C.c_float(wd), C.c_int64(step))
    if rc != 0:
        raise ValueError("oracle_zero1_adamw failed")
    return params
