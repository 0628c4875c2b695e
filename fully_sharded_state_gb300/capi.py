"""Thin ctypes binding of the shard engine's C ABI (``include/fsdp_shard.h``).

Argument marshalling only: every step of the data path runs in the CUDA
library. Functions keep the C names. Buffers are torch tensors on a CUDA
device (torch provides memory and streams); each "per-rank" argument is a
list of R tensors. A missing library raises ``LibraryNotBuilt``: there is no
fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libfsdp_shard.so")

FSDP_OK, FSDP_EINVAL, FSDP_EALIGN, FSDP_ERANGE, FSDP_ECUDA, FSDP_EUNSUPPORTED = 0, -1, -2, -3, -4, -5
FSDP_FLAT, FSDP_PER_PARAM, FSDP_ZERO3 = 1, 2, 3
FSDP_F32, FSDP_BF16 = 0, 1
FSDP_MAX_RANKS = 64
FSDP_SEG_ALIGN = 8

(Q_FULL_NUMEL, Q_SHARD_NUMEL, Q_PADDED_NUMEL, Q_N_PARAMS, Q_RANKS, Q_MODE, Q_PARAM_DTYPE,
 Q_GRAD_DTYPE, Q_PARAM_FULL_OFFSET, Q_PARAM_SHARD_OFFSET, Q_PARAM_SHARD_ROWS,
 Q_PARAM_RANK_ROW_START, Q_PARAM_RANK_ROWS, Q_RANK_NUMEL, Q_PARAM_OWNER) = range(15)

_STATUS_NAMES = {0: "FSDP_OK", -1: "FSDP_EINVAL", -2: "FSDP_EALIGN", -3: "FSDP_ERANGE",
                 -4: "FSDP_ECUDA", -5: "FSDP_EUNSUPPORTED"}


class LibraryNotBuilt(RuntimeError):
    pass


class FsdpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class AdamWHP(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double)]


_lib = None
_vp = ctypes.c_void_p
_i64p = ctypes.POINTER(ctypes.c_int64)


def load(path: str = LIB_PATH):
    """Load the CUDA library (built by ``fully_sharded_state_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise LibraryNotBuilt(
            f"{path} is missing: build it with `python -m fully_sharded_state_gb300.build` "
            "(or __graft_entry__.build()); the shard engine has no non-CUDA fallback")
    L = ctypes.CDLL(path)
    L.fsdp_layout.restype = ctypes.c_int
    L.fsdp_layout.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _i64p, _i64p,
                              ctypes.c_int, ctypes.c_int, ctypes.POINTER(_vp)]
    L.fsdp_layout_destroy.restype = None
    L.fsdp_layout_destroy.argtypes = [_vp]
    L.fsdp_layout_query.restype = ctypes.c_int
    L.fsdp_layout_query.argtypes = [_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i64p]
    L.fsdp_pack_flat.restype = ctypes.c_int
    L.fsdp_pack_flat.argtypes = [_vp, _vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp]
    L.fsdp_all_gather_unflatten.restype = ctypes.c_int
    L.fsdp_all_gather_unflatten.argtypes = [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp]
    L.fsdp_reduce_scatter_adamw.restype = ctypes.c_int
    L.fsdp_reduce_scatter_adamw.argtypes = [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                            ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                            ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                            ctypes.POINTER(AdamWHP), ctypes.c_int64, _vp]
    L.fsdp_reduce_scatter_adamw_gather.restype = ctypes.c_int
    L.fsdp_reduce_scatter_adamw_gather.argtypes = [
        _vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
        ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(AdamWHP), ctypes.c_int64,
        _vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp]
    L.fsdp_all_reduce.restype = ctypes.c_int
    L.fsdp_all_reduce.argtypes = [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.c_int, _vp]
    L.fsdp_accumulate_grad.restype = ctypes.c_int
    L.fsdp_accumulate_grad.argtypes = [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.c_int,
                                       _vp]
    L.fsdp_reduce_scatter_adamw_accum.restype = ctypes.c_int
    L.fsdp_reduce_scatter_adamw_accum.argtypes = [
        _vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
        ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(AdamWHP),
        ctypes.c_int64, _vp]
    L.fsdp_last_error.restype = ctypes.c_char_p
    L.fsdp_last_error.argtypes = []
    L.fsdp_version.restype = ctypes.c_char_p
    L.fsdp_version.argtypes = []
    _lib = L
    return L


def _check(status: int) -> None:
    if status != FSDP_OK:
        raise FsdpError(status, load().fsdp_last_error().decode())


def _dims(shapes):
    d0, inner = [], []
    for shp in shapes:
        shp = tuple(int(x) for x in shp)
        d0.append(shp[0] if shp else 1)
        n = 1
        for x in shp[1:]:
            n *= x
        inner.append(n)
    return d0, inner


class Layout:
    """Owns one ``fsdp_layout_t``. Query helpers mirror ``fsdp_layout_query``."""

    def __init__(self, handle, mode, R, shapes, param_dtype, grad_dtype):
        self._h = handle
        self.mode, self.R, self.shapes = mode, R, [tuple(s) for s in shapes]
        self.param_dtype, self.grad_dtype = param_dtype, grad_dtype

    @property
    def handle(self):
        return self._h

    def query(self, what: int, i: int = 0, r: int = 0) -> int:
        out = ctypes.c_int64(0)
        _check(load().fsdp_layout_query(self._h, what, i, r, ctypes.byref(out)))
        return out.value

    @property
    def full_numel(self) -> int:
        return self.query(Q_FULL_NUMEL)

    @property
    def shard_numel(self) -> int:
        return self.query(Q_SHARD_NUMEL)

    def param_full_offset(self, i: int) -> int:
        return self.query(Q_PARAM_FULL_OFFSET, i)

    def param_shard_offset(self, i: int) -> int:
        return self.query(Q_PARAM_SHARD_OFFSET, i)

    def rank_rows(self, i: int, r: int):
        return self.query(Q_PARAM_RANK_ROW_START, i, r), self.query(Q_PARAM_RANK_ROWS, i, r)

    def rank_numel(self, r: int) -> int:
        return self.query(Q_RANK_NUMEL, 0, r)

    def param_owner(self, i: int) -> int:
        """ZeRO-3 layouts: the rank that holds parameter i whole."""
        return self.query(Q_PARAM_OWNER, i)

    def close(self):
        if self._h:
            load().fsdp_layout_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fsdp_layout(mode: int, R: int, shapes, param_dtype: int, grad_dtype: int) -> Layout:
    """Build the layout of one FSDP unit (see ``fsdp_layout`` in the header)."""
    d0, inner = _dims(shapes)
    n = len(d0)
    a0 = (ctypes.c_int64 * max(1, n))(*d0)
    a1 = (ctypes.c_int64 * max(1, n))(*inner)
    h = _vp()
    _check(load().fsdp_layout(mode, R, n, a0, a1, param_dtype, grad_dtype, ctypes.byref(h)))
    return Layout(h, mode, R, shapes, param_dtype, grad_dtype)


def _ptr_array(tensors, R, name, allow_none=False):
    if tensors is None:
        if allow_none:
            return None
        raise ValueError(f"{name}: expected {R} tensors, got None")
    if len(tensors) != R:
        raise ValueError(f"{name}: expected {R} tensors, got {len(tensors)}")
    arr = (_vp * R)()
    for r, t in enumerate(tensors):
        if not t.is_cuda:
            raise ValueError(f"{name}[{r}] is not a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name}[{r}] is not contiguous")
        arr[r] = t.data_ptr()
    return arr


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return _vp(stream.cuda_stream)


def fsdp_pack_flat(layout: Layout, full, param_shard, master, stream=None) -> None:
    """Shard the full fp32 unit into every rank's master (and bf16) buffer."""
    R = layout.R
    if not full.is_cuda or not full.is_contiguous():
        raise ValueError("full must be a contiguous CUDA tensor")
    ps = _ptr_array(param_shard, R, "param_shard", allow_none=True)
    ms = _ptr_array(master, R, "master")
    _check(load().fsdp_pack_flat(layout.handle, _vp(full.data_ptr()), ps, ms,
                                 _stream_handle(stream)))


def fsdp_all_gather_unflatten(layout: Layout, shard, full_out, stream=None) -> None:
    """Rebuild every destination rank's full unit from the R shard buffers."""
    R = layout.R
    _check(load().fsdp_all_gather_unflatten(layout.handle, _ptr_array(shard, R, "shard"),
                                            _ptr_array(full_out, R, "full_out"),
                                            _stream_handle(stream)))


def fsdp_reduce_scatter_adamw(layout: Layout, grad_full, master, m, v, param_shard_out,
                              grad_shard_out, hp: AdamWHP, step: int, stream=None) -> None:
    """Fixed-order fp32 reduce-scatter fused with the sharded AdamW step."""
    R = layout.R
    _check(load().fsdp_reduce_scatter_adamw(
        layout.handle, _ptr_array(grad_full, R, "grad_full"), _ptr_array(master, R, "master"),
        _ptr_array(m, R, "m"), _ptr_array(v, R, "v"),
        _ptr_array(param_shard_out, R, "param_shard_out", allow_none=True),
        _ptr_array(grad_shard_out, R, "grad_shard_out", allow_none=True),
        ctypes.byref(hp), int(step), _stream_handle(stream)))


def fsdp_reduce_scatter_adamw_gather(layout: Layout, grad_full, master, m, v, param_shard_out,
                                     grad_shard_out, hp: AdamWHP, step: int,
                                     gather_layout: Layout, shard, full_out, stream=None) -> None:
    """Reduce-scatter + AdamW of one unit, then the all-gather of another (prefetch)."""
    R, G = layout.R, gather_layout.R
    _check(load().fsdp_reduce_scatter_adamw_gather(
        layout.handle, _ptr_array(grad_full, R, "grad_full"), _ptr_array(master, R, "master"),
        _ptr_array(m, R, "m"), _ptr_array(v, R, "v"),
        _ptr_array(param_shard_out, R, "param_shard_out", allow_none=True),
        _ptr_array(grad_shard_out, R, "grad_shard_out", allow_none=True),
        ctypes.byref(hp), int(step), gather_layout.handle, _ptr_array(shard, G, "shard"),
        _ptr_array(full_out, G, "full_out"), _stream_handle(stream)))


def fsdp_all_reduce(layout: Layout, grad_full, out, out_dtype: int, stream=None) -> None:
    """DDP all-reduce: every rank's output gets the fixed-order average."""
    R = layout.R
    _check(load().fsdp_all_reduce(layout.handle, _ptr_array(grad_full, R, "grad_full"),
                                  _ptr_array(out, R, "out"), int(out_dtype),
                                  _stream_handle(stream)))


def fsdp_accumulate_grad(layout: Layout, acc_full, grad_full, first: bool, stream=None) -> None:
    """Add one micro-batch's gradients into the R fp32 accumulators (copy if first)."""
    R = layout.R
    _check(load().fsdp_accumulate_grad(layout.handle, _ptr_array(acc_full, R, "acc_full"),
                                       _ptr_array(grad_full, R, "grad_full"), int(bool(first)),
                                       _stream_handle(stream)))


def fsdp_reduce_scatter_adamw_accum(layout: Layout, acc_full, grad_full, master, m, v,
                                    param_shard_out, grad_shard_out, hp: AdamWHP, step: int,
                                    stream=None) -> None:
    """The last micro-batch fused into reduce-scatter + AdamW."""
    R = layout.R
    _check(load().fsdp_reduce_scatter_adamw_accum(
        layout.handle, _ptr_array(acc_full, R, "acc_full"), _ptr_array(grad_full, R, "grad_full"),
        _ptr_array(master, R, "master"), _ptr_array(m, R, "m"), _ptr_array(v, R, "v"),
        _ptr_array(param_shard_out, R, "param_shard_out", allow_none=True),
        _ptr_array(grad_shard_out, R, "grad_shard_out", allow_none=True),
        ctypes.byref(hp), int(step), _stream_handle(stream)))


def fsdp_version() -> str:
    return load().fsdp_version().decode()
