"""fsdp_sharded_state_gb300 -- the FSDP / ZeRO-3 sharded-state step on one GB300.

Thin ctypes binding of ``libfsdpstate.so`` (C ABI in ``include/fsdp_state.h``).
The functions here carry the C names and only marshal arguments: torch tensors
(or raw device pointers) in, status codes checked, ``FsdpError`` out.  Every step
of the path runs in the library's CUDA kernels; there is no CPU fallback -- if the
library is missing, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libfsdpstate.so")

FSDP_FLAT, FSDP_DIM0, FSDP_ZERO1 = 0, 1, 2
FSDP_F32, FSDP_BF16 = 0, 1
MODES = {"flat": FSDP_FLAT, "dim0": FSDP_DIM0, "zero1": FSDP_ZERO1}

FSDP_RS_AUTO, FSDP_RS_DIRECT, FSDP_RS_STAGED = 0, 1, 2
RS_KERNELS = {"auto": FSDP_RS_AUTO, "direct": FSDP_RS_DIRECT, "staged": FSDP_RS_STAGED}

FSDP_OK = 0
STATUS = {0: "FSDP_OK", -1: "FSDP_EINVAL", -2: "FSDP_EDTYPE", -3: "FSDP_ESHAPE", -4: "FSDP_EALIGN",
          -5: "FSDP_EOVERFLOW", -6: "FSDP_ECUDA", -7: "FSDP_ETIMEOUT", -8: "FSDP_ENOMEM"}

# Every symbol include/fsdp_state.h declares.
EXPORTS = ("fsdp_layout_create", "fsdp_layout_destroy", "fsdp_layout_query", "fsdp_layout_unit",
           "fsdp_layout_tensor", "fsdp_layout_segment", "fsdp_state_bytes", "fsdp_layout_prepare",
           "fsdp_unshard", "fsdp_reduce_scatter_adamw", "fsdp_reshard", "fsdp_check_status",
           "fsdp_error_string", "fsdp_last_cuda_error", "fsdp_reduce_scatter_adamw_noalloc",
           "fsdp_layout_owner", "fsdp_clip_workspace_bytes", "fsdp_reduce_scatter_clip_adamw",
           "fsdp_accumulate_grads", "fsdp_hsdp_reduce_scatter_adamw", "fsdp_zero1_adamw_broadcast",
           "fsdp_set_rs_kernel", "fsdp_rs_kernel_for", "fsdp_wait_selftest", "fsdp_adamw_step_consts_make",
           "fsdp_reduce_scatter_adamw_consts", "fsdp_adamw_step_consts_upload", "fsdp_collective_payload",
           "fsdp_accumulate_reduce_scatter_adamw")


class FsdpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)}"
        if status == -6 and _lib is not None:
            msg += f" ({_lib.fsdp_last_cuda_error().decode()})"
        super().__init__(msg)


class LayoutInfo(C.Structure):
    _fields_ = [("n_tensors", C.c_int32), ("n_units", C.c_int32), ("n_ranks", C.c_int32), ("mode", C.c_int32),
                ("numel", C.c_int64), ("shard_numel", C.c_int64), ("shard_stride", C.c_int64),
                ("full_numel", C.c_int64), ("pad_numel", C.c_int64), ("n_segments", C.c_int64)]


FSDP_NO_SHARD, FSDP_ZERO1_OPT, FSDP_SHARD_GRAD_OP, FSDP_FULL_SHARD, FSDP_HYBRID_SHARD = 0, 1, 2, 3, 4
STRATEGIES = {"no_shard": FSDP_NO_SHARD, "zero1": FSDP_ZERO1_OPT, "shard_grad_op": FSDP_SHARD_GRAD_OP,
              "full_shard": FSDP_FULL_SHARD, "hybrid_shard": FSDP_HYBRID_SHARD}


class CollectivePayload(C.Structure):
    _fields_ = [("allreduce_input", C.c_int64), ("forward_allgather", C.c_int64),
                ("backward_allgather", C.c_int64), ("reducescatter_input", C.c_int64), ("broadcast", C.c_int64),
                ("bus_elements", C.c_double)]


class AdamWHparams(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("weight_decay", C.c_float)]


class AdamWStepConsts(C.Structure):
    """The 48-byte block of per-step AdamW constants (fsdp_adamw_step_consts)."""
    _fields_ = [("decay", C.c_float), ("om1", C.c_float), ("om2", C.c_float), ("step_size", C.c_float),
                ("bc2s", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("n_avg", C.c_float), ("reserved", C.c_float * 3)]


_lib: Optional[C.CDLL] = None


def lib() -> C.CDLL:
    """The loaded libfsdpstate; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libfsdpstate is not built ({LIB_PATH} missing): run "
                               "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = C.CDLL(LIB_PATH)
        vp, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
        L.fsdp_layout_create.argtypes = [i32, vp, vp, vp, vp, i32, i32, C.POINTER(vp)]
        L.fsdp_layout_destroy.argtypes = [vp]
        L.fsdp_layout_destroy.restype = None
        L.fsdp_layout_query.argtypes = [vp, C.POINTER(LayoutInfo)]
        L.fsdp_layout_unit.argtypes = [vp, i32] + [C.POINTER(i64)] * 5
        L.fsdp_layout_tensor.argtypes = [vp, i32, C.POINTER(i32)] + [C.POINTER(i64)] * 4
        L.fsdp_layout_segment.argtypes = [vp, i32, i32] + [C.POINTER(i64)] * 4
        L.fsdp_state_bytes.argtypes = [vp, i32, i32, i32, i64, i64, i64, i64, C.POINTER(i64)]
        L.fsdp_collective_payload.argtypes = [vp, i32, i32, C.POINTER(CollectivePayload)]
        L.fsdp_layout_prepare.argtypes = [vp]
        L.fsdp_unshard.argtypes = [vp, i32, i32, vp, vp, i32, vp]
        L.fsdp_reduce_scatter_adamw.argtypes = [vp, i32, i32, C.POINTER(vp), i32, vp, vp, vp, vp, vp,
                                                C.POINTER(AdamWHparams), i64, vp]
        L.fsdp_reshard.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp]
        L.fsdp_reduce_scatter_adamw_noalloc.argtypes = L.fsdp_reduce_scatter_adamw.argtypes
        L.fsdp_layout_owner.argtypes = [vp, i32, C.POINTER(i32)]
        L.fsdp_clip_workspace_bytes.argtypes = []
        L.fsdp_clip_workspace_bytes.restype = C.c_size_t
        L.fsdp_reduce_scatter_clip_adamw.argtypes = [vp, i32, i32, C.POINTER(vp), i32, vp, vp, vp, vp, vp, C.c_float,
                                                     vp, vp, C.POINTER(AdamWHparams), i64, vp]
        L.fsdp_accumulate_grads.argtypes = [vp, i32, i32, C.POINTER(vp), C.POINTER(vp), i32, i32, vp]
        L.fsdp_accumulate_reduce_scatter_adamw.argtypes = [vp, i32, i32, C.POINTER(vp), C.POINTER(vp), i32, vp, vp,
                                                           vp, vp, vp, C.POINTER(AdamWHparams), i64, vp]
        L.fsdp_hsdp_reduce_scatter_adamw.argtypes = [vp, i32, i32, i32, C.POINTER(vp), i32, vp, vp, vp, vp,
                                                     C.POINTER(AdamWHparams), i64, vp]
        L.fsdp_zero1_adamw_broadcast.argtypes = [vp, i32, i32, C.POINTER(vp), i32, vp, vp, vp, C.POINTER(vp), i32,
                                                 C.POINTER(AdamWHparams), i64, vp]
        L.fsdp_check_status.argtypes = [vp]
        L.fsdp_set_rs_kernel.argtypes = [i32]
        L.fsdp_rs_kernel_for.argtypes = [vp, i32]
        L.fsdp_wait_selftest.argtypes = [i64, vp]
        L.fsdp_adamw_step_consts_make.argtypes = [vp, C.POINTER(AdamWHparams), i64, C.POINTER(AdamWStepConsts)]
        L.fsdp_reduce_scatter_adamw_consts.argtypes = [vp, i32, i32, C.POINTER(vp), i32, vp, vp, vp, vp, vp, vp, vp]
        L.fsdp_adamw_step_consts_upload.argtypes = [vp, vp, vp]
        L.fsdp_error_string.argtypes = [C.c_int]
        L.fsdp_error_string.restype = C.c_char_p
        L.fsdp_last_cuda_error.argtypes = []
        L.fsdp_last_cuda_error.restype = C.c_char_p
        _lib = L
    return _lib


def _check(rc: int, where: str) -> None:
    if rc != FSDP_OK:
        raise FsdpError(rc, where)


def _ptr(x) -> Optional[int]:
    """Device address of a tensor (or an int address); None stays NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("buffers must be contiguous")
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return FSDP_F32
    if t.dtype == torch.bfloat16:
        return FSDP_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: float32 or bfloat16")


class Layout:
    """An fsdp_layout: shapes + unit ids + N + mode -> offsets, padding, segments."""

    def __init__(self, shapes: Sequence[Sequence[int]], unit_ids: Optional[Sequence[int]] = None,
                 n_ranks: int = 1, mode: int = FSDP_FLAT, dtypes: Optional[Sequence[int]] = None):
        shapes = [tuple(int(d) for d in s) for s in shapes]
        T = len(shapes)
        if unit_ids is None:
            unit_ids = [0] * T
        ndim = (C.c_int32 * max(T, 1))(*[len(s) for s in shapes])
        flat = [d for s in shapes for d in s] or [0]
        dims = (C.c_int64 * len(flat))(*flat)
        units = (C.c_int32 * max(T, 1))(*unit_ids)
        dt = None if dtypes is None else (C.c_int32 * max(T, 1))(*dtypes)
        h = C.c_void_p()
        self._h = None
        _check(lib().fsdp_layout_create(T, ndim, dims, units, dt, n_ranks, mode, C.byref(h)),
               "fsdp_layout_create")
        self._h = h
        self.shapes, self.unit_ids, self.n_ranks, self.mode = shapes, list(unit_ids), n_ranks, mode
        info = LayoutInfo()
        _check(lib().fsdp_layout_query(self._h, C.byref(info)), "fsdp_layout_query")
        self.info = {k: getattr(info, k) for k, _ in LayoutInfo._fields_}

    # -- queries --------------------------------------------------------------
    @property
    def handle(self):
        return self._h

    @property
    def N(self) -> int:
        return self.info["n_ranks"]

    @property
    def stride(self) -> int:
        return self.info["shard_stride"]

    @property
    def n_units(self) -> int:
        return self.info["n_units"]

    def unit(self, u: int) -> dict:
        v = [C.c_int64() for _ in range(5)]
        _check(lib().fsdp_layout_unit(self._h, u, *[C.byref(x) for x in v]), "fsdp_layout_unit")
        return dict(zip(("shard_off", "shard_numel", "full_off", "full_numel", "numel"), (x.value for x in v)))

    def tensor(self, t: int) -> dict:
        u = C.c_int32()
        v = [C.c_int64() for _ in range(4)]
        _check(lib().fsdp_layout_tensor(self._h, t, C.byref(u), *[C.byref(x) for x in v]), "fsdp_layout_tensor")
        d = dict(zip(("numel", "full_off", "shard_off", "rows_per_rank"), (x.value for x in v)))
        d["unit"] = u.value
        return d

    def segment(self, t: int, r: int) -> dict:
        v = [C.c_int64() for _ in range(4)]
        _check(lib().fsdp_layout_segment(self._h, t, r, *[C.byref(x) for x in v]), "fsdp_layout_segment")
        return dict(zip(("shard_off", "full_off", "len", "pad"), (x.value for x in v)))

    def owner(self, t: int) -> int:
        r = C.c_int32()
        _check(lib().fsdp_layout_owner(self._h, t, C.byref(r)), "fsdp_layout_owner")
        return r.value

    def state_bytes(self, stage: int, rank: int, physical: bool, param_bytes: int, grad_bytes: int,
                    optim_bytes: int, step_bytes: int = 0):
        out = (C.c_int64 * 3)()
        _check(lib().fsdp_state_bytes(self._h, stage, rank, int(physical), param_bytes, grad_bytes, optim_bytes,
                                      step_bytes, out), "fsdp_state_bytes")
        return tuple(out)

    def collective_payload(self, strategy, n_groups: int = 1) -> dict:
        """Per-rank collective payload of one step (fsdp_collective_payload): logical
        input elements of each collective and the ring bus elements a rank sends."""
        code = STRATEGIES[strategy] if isinstance(strategy, str) else int(strategy)
        out = CollectivePayload()
        _check(lib().fsdp_collective_payload(self._h, code, n_groups, C.byref(out)), "fsdp_collective_payload")
        return {f: getattr(out, f) for f, _ in CollectivePayload._fields_}

    def prepare(self) -> None:
        _check(lib().fsdp_layout_prepare(self._h), "fsdp_layout_prepare")

    def close(self) -> None:
        if self._h is not None and _lib is not None:
            _lib.fsdp_layout_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# -- the C names ----------------------------------------------------------------
def fsdp_layout_create(shapes, unit_ids=None, n_ranks=1, mode=FSDP_FLAT, dtypes=None) -> Layout:
    return Layout(shapes, unit_ids, n_ranks, mode, dtypes)


def fsdp_unshard(layout: Layout, unit_begin: int, unit_end: int, param_shards, full, stream=None,
                 elem_dtype: Optional[int] = None) -> None:
    if elem_dtype is None:
        elem_dtype = _dtype_code(param_shards)
    _check(lib().fsdp_unshard(layout.handle, unit_begin, unit_end, _ptr(param_shards), _ptr(full), elem_dtype,
                              _stream(stream)), "fsdp_unshard")


def fsdp_reduce_scatter_adamw(layout: Layout, unit_begin: int, unit_end: int, grad_replicas, master, exp_avg,
                              exp_avg_sq, param_shards=None, grad_shard_out=None,
                              hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step: int = 1, stream=None,
                              grad_dtype: Optional[int] = None) -> None:
    if len(grad_replicas) != layout.N:
        raise ValueError(f"need {layout.N} gradient replicas, got {len(grad_replicas)}")
    if grad_dtype is None:
        grad_dtype = _dtype_code(grad_replicas[0])
    arr = (C.c_void_p * layout.N)(*[_ptr(g) for g in grad_replicas])
    h = hp if isinstance(hp, AdamWHparams) else AdamWHparams(*hp)
    _check(lib().fsdp_reduce_scatter_adamw(layout.handle, unit_begin, unit_end, arr, grad_dtype, _ptr(master),
                                           _ptr(exp_avg), _ptr(exp_avg_sq), _ptr(param_shards),
                                           _ptr(grad_shard_out), C.byref(h), step, _stream(stream)),
           "fsdp_reduce_scatter_adamw")


def fsdp_reduce_scatter_adamw_noalloc(layout: Layout, unit_begin: int, unit_end: int, grad_replicas, master,
                                      exp_avg, exp_avg_sq, param_shards=None, grad_shard_out=None,
                                      hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step: int = 1, stream=None,
                                      grad_dtype: Optional[int] = None) -> None:
    """fsdp_reduce_scatter_adamw without any device allocation (fixed in-library scratch)."""
    if len(grad_replicas) != layout.N:
        raise ValueError(f"need {layout.N} gradient replicas, got {len(grad_replicas)}")
    if grad_dtype is None:
        grad_dtype = _dtype_code(grad_replicas[0])
    arr = (C.c_void_p * layout.N)(*[_ptr(g) for g in grad_replicas])
    h = hp if isinstance(hp, AdamWHparams) else AdamWHparams(*hp)
    _check(lib().fsdp_reduce_scatter_adamw_noalloc(layout.handle, unit_begin, unit_end, arr, grad_dtype,
                                                   _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
                                                   _ptr(param_shards), _ptr(grad_shard_out), C.byref(h), step,
                                                   _stream(stream)), "fsdp_reduce_scatter_adamw_noalloc")


def fsdp_adamw_step_consts_make(layout: Layout, hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step: int = 1) -> AdamWStepConsts:
    """The step's AdamW constants as the fused step forms them (host only)."""
    out = AdamWStepConsts()
    h = hp if isinstance(hp, AdamWHparams) else AdamWHparams(*hp)
    _check(lib().fsdp_adamw_step_consts_make(layout.handle, C.byref(h), step, C.byref(out)),
           "fsdp_adamw_step_consts_make")
    return out


def fsdp_adamw_step_consts_upload(dev_dst, host_src, stream=None) -> None:
    """Copies a 48-byte block of step constants from (pinned) host memory to the device
    block on the stream; inside a CUDA graph capture it reads host_src at every replay."""
    _check(lib().fsdp_adamw_step_consts_upload(_ptr(dev_dst), _ptr(host_src), _stream(stream)),
           "fsdp_adamw_step_consts_upload")


def fsdp_reduce_scatter_adamw_consts(layout: Layout, unit_begin: int, unit_end: int, grad_replicas, master,
                                     exp_avg, exp_avg_sq, param_shards=None, grad_shard_out=None, consts=None,
                                     stream=None, grad_dtype: Optional[int] = None) -> None:
    """fsdp_reduce_scatter_adamw with the step constants read on the device from `consts`
    (a 48-byte device buffer, e.g. a float32 tensor of 12 elements)."""
    if len(grad_replicas) != layout.N:
        raise ValueError(f"need {layout.N} gradient replicas, got {len(grad_replicas)}")
    if grad_dtype is None:
        grad_dtype = _dtype_code(grad_replicas[0])
    arr = (C.c_void_p * layout.N)(*[_ptr(g) for g in grad_replicas])
    _check(lib().fsdp_reduce_scatter_adamw_consts(layout.handle, unit_begin, unit_end, arr, grad_dtype,
                                                  _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
                                                  _ptr(param_shards), _ptr(grad_shard_out), _ptr(consts),
                                                  _stream(stream)), "fsdp_reduce_scatter_adamw_consts")


def _ptr_array(xs):
    return (C.c_void_p * len(xs))(*[_ptr(x) for x in xs])


def _hp(hp):
    return hp if isinstance(hp, AdamWHparams) else AdamWHparams(*hp)


def fsdp_clip_workspace_bytes() -> int:
    return int(lib().fsdp_clip_workspace_bytes())


def fsdp_reduce_scatter_clip_adamw(layout: Layout, unit_begin: int, unit_end: int, grad_replicas, master, exp_avg,
                                   exp_avg_sq, param_shards, grad_shard, max_norm: float, workspace,
                                   norm_out=None, hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step: int = 1,
                                   stream=None, grad_dtype: Optional[int] = None) -> None:
    if len(grad_replicas) != layout.N:
        raise ValueError(f"need {layout.N} gradient replicas, got {len(grad_replicas)}")
    if grad_dtype is None:
        grad_dtype = _dtype_code(grad_replicas[0])
    _check(lib().fsdp_reduce_scatter_clip_adamw(layout.handle, unit_begin, unit_end, _ptr_array(grad_replicas),
                                                grad_dtype, _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
                                                _ptr(param_shards), _ptr(grad_shard), float(max_norm),
                                                _ptr(workspace), _ptr(norm_out), C.byref(_hp(hp)), step,
                                                _stream(stream)), "fsdp_reduce_scatter_clip_adamw")


def fsdp_accumulate_grads(layout: Layout, unit_begin: int, unit_end: int, acc, micro, first: bool,
                          stream=None, micro_dtype: Optional[int] = None) -> None:
    if len(acc) != layout.N or len(micro) != layout.N:
        raise ValueError(f"need {layout.N} accumulators and micro-gradients")
    if micro_dtype is None:
        micro_dtype = _dtype_code(micro[0])
    _check(lib().fsdp_accumulate_grads(layout.handle, unit_begin, unit_end, _ptr_array(acc), _ptr_array(micro),
                                       micro_dtype, int(bool(first)), _stream(stream)), "fsdp_accumulate_grads")


def fsdp_accumulate_reduce_scatter_adamw(layout: Layout, unit_begin: int, unit_end: int, acc, micro, master,
                                         exp_avg, exp_avg_sq, param_shards=None, grad_shard_out=None,
                                         hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step: int = 1, stream=None,
                                         micro_dtype: Optional[int] = None) -> None:
    """The last micro-batch of a no_sync accumulation fused with the step: acc (N fp32
    accumulators, read only) plus micro (N micro-batch gradients), reduce-scattered, AdamW, cast."""
    if len(acc) != layout.N or len(micro) != layout.N:
        raise ValueError(f"need {layout.N} accumulators and micro-gradients")
    if micro_dtype is None:
        micro_dtype = _dtype_code(micro[0])
    h = hp if isinstance(hp, AdamWHparams) else AdamWHparams(*hp)
    _check(lib().fsdp_accumulate_reduce_scatter_adamw(layout.handle, unit_begin, unit_end, _ptr_array(acc),
                                                      _ptr_array(micro), micro_dtype, _ptr(master), _ptr(exp_avg),
                                                      _ptr(exp_avg_sq), _ptr(param_shards), _ptr(grad_shard_out),
                                                      C.byref(h), step, _stream(stream)),
           "fsdp_accumulate_reduce_scatter_adamw")


def fsdp_hsdp_reduce_scatter_adamw(layout: Layout, unit_begin: int, unit_end: int, n_groups: int, grad_replicas,
                                   master, exp_avg, exp_avg_sq, param_shards=None,
                                   hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step: int = 1, stream=None,
                                   grad_dtype: Optional[int] = None) -> None:
    if len(grad_replicas) != layout.N * n_groups:
        raise ValueError(f"need {layout.N * n_groups} gradient replicas, got {len(grad_replicas)}")
    if grad_dtype is None:
        grad_dtype = _dtype_code(grad_replicas[0])
    _check(lib().fsdp_hsdp_reduce_scatter_adamw(layout.handle, unit_begin, unit_end, n_groups,
                                                _ptr_array(grad_replicas), grad_dtype, _ptr(master), _ptr(exp_avg),
                                                _ptr(exp_avg_sq), _ptr(param_shards), C.byref(_hp(hp)), step,
                                                _stream(stream)), "fsdp_hsdp_reduce_scatter_adamw")


def fsdp_zero1_adamw_broadcast(layout: Layout, unit_begin: int, unit_end: int, grad_replicas, master, exp_avg,
                               exp_avg_sq, param_replicas, hp=(1e-3, 0.9, 0.999, 1e-8, 0.01), step: int = 1,
                               stream=None, grad_dtype: Optional[int] = None,
                               param_dtype: Optional[int] = None) -> None:
    if len(grad_replicas) != layout.N or len(param_replicas) != layout.N:
        raise ValueError(f"need {layout.N} gradient and parameter replicas")
    if grad_dtype is None:
        grad_dtype = _dtype_code(grad_replicas[0])
    if param_dtype is None:
        param_dtype = _dtype_code(param_replicas[0])
    _check(lib().fsdp_zero1_adamw_broadcast(layout.handle, unit_begin, unit_end, _ptr_array(grad_replicas),
                                            grad_dtype, _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
                                            _ptr_array(param_replicas), param_dtype, C.byref(_hp(hp)), step,
                                            _stream(stream)), "fsdp_zero1_adamw_broadcast")


def fsdp_reshard(layout: Layout, unit_begin: int, unit_end: int, full=None, master=None, param_shards=None,
                 stream=None, full_dtype: Optional[int] = None) -> None:
    if full is not None and full_dtype is None:
        full_dtype = _dtype_code(full)
    _check(lib().fsdp_reshard(layout.handle, unit_begin, unit_end, _ptr(full), full_dtype or 0, _ptr(master),
                              _ptr(param_shards), _stream(stream)), "fsdp_reshard")


def fsdp_check_status(stream=None) -> None:
    _check(lib().fsdp_check_status(_stream(stream)), "fsdp_check_status")


def fsdp_set_rs_kernel(kind) -> int:
    """Selects the kernel of fsdp_reduce_scatter_adamw ("auto", "direct", "staged"
    or the FSDP_RS_* code); returns the previous code."""
    code = RS_KERNELS[kind] if isinstance(kind, str) else int(kind)
    prev = lib().fsdp_set_rs_kernel(code)
    if prev < 0:
        raise FsdpError(prev, "fsdp_set_rs_kernel")
    return prev


def fsdp_rs_kernel_for(layout: Layout, grad_dtype) -> str:
    """"direct" or "staged": the kernel fsdp_reduce_scatter_adamw runs for this
    layout and gradient dtype (a torch dtype or FSDP_F32/FSDP_BF16) right now."""
    import torch
    code = grad_dtype if isinstance(grad_dtype, int) else {torch.float32: FSDP_F32, torch.bfloat16: FSDP_BF16}[grad_dtype]
    rc = lib().fsdp_rs_kernel_for(layout.handle, code)
    if rc < 0:
        raise FsdpError(rc, "fsdp_rs_kernel_for")
    return {FSDP_RS_DIRECT: "direct", FSDP_RS_STAGED: "staged"}[rc]


def fsdp_wait_selftest(timeout_ns: int, stream=None) -> None:
    _check(lib().fsdp_wait_selftest(int(timeout_ns), _stream(stream)), "fsdp_wait_selftest")


def fsdp_error_string(status: int) -> str:
    return lib().fsdp_error_string(status).decode()


from .state import ShardedState, StepGraph, step_schedule  # noqa: E402  (harness over the calls above)
from .hostfeed import HostFeed  # noqa: E402  (host-fed steps over ShardedState)
