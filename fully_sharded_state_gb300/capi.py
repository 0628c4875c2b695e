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


class FsdpArgumentError(FsdpError, ValueError):
    """A tensor argument that does not fit the layout (count, device, dtype,
    size, contiguity), caught by the binding before the C call."""

    def __init__(self, message: str):
        super().__init__(FSDP_EINVAL, message)


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
    L.fsdp_all_gather_unflatten_units.restype = ctypes.c_int
    L.fsdp_all_gather_unflatten_units.argtypes = [ctypes.c_int, ctypes.POINTER(_vp),
                                                  ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp]
    L.fsdp_reduce_scatter_adamw_units.restype = ctypes.c_int
    L.fsdp_reduce_scatter_adamw_units.argtypes = [
        ctypes.c_int, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
        ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
        ctypes.POINTER(AdamWHP), ctypes.c_int64, _vp]
    L.fsdp_write_stream.restype = ctypes.c_int
    L.fsdp_write_stream.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, ctypes.c_int64,
                                    ctypes.c_uint32, _vp]
    L.fsdp_adamw_from_reduced.restype = ctypes.c_int
    L.fsdp_adamw_from_reduced.argtypes = [_vp] + [ctypes.POINTER(_vp)] * 5 + [
        ctypes.POINTER(AdamWHP), ctypes.c_int64, _vp]
    L.fsdp_stage_wait_timeouts.restype = ctypes.c_int
    L.fsdp_stage_wait_timeouts.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint64)]
    L.fsdp_stage_wait_selftest.restype = ctypes.c_int
    L.fsdp_stage_wait_selftest.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint64)]
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


_TORCH_DTYPES = {}


def _torch_dtype(fsdp_dtype: int):
    import torch
    if not _TORCH_DTYPES:
        _TORCH_DTYPES.update({FSDP_BF16: torch.bfloat16, FSDP_F32: torch.float32})
    return _TORCH_DTYPES[fsdp_dtype]


class _Args:
    """Marshals the tensor arguments of one call into C pointer arrays, after
    checking each tensor against what the layout says it must hold: the
    count of tensors, a CUDA tensor on the call's one device, contiguous,
    the dtype, and at least the number of elements the kernels touch. The
    C library can only check pointers (NULL, alignment, overlap, device
    memory of one device), so these checks keep a short or mistyped tensor
    from reaching a kernel."""

    def __init__(self):
        self.device = None

    def one(self, t, name: str, numel: int, dtype: int):
        if not getattr(t, "is_cuda", False):
            raise FsdpArgumentError(f"{name} is not a CUDA tensor")
        dev = t.device
        if self.device is None:
            self.device = dev
        elif dev != self.device:
            raise FsdpArgumentError(f"{name} is on {dev}, the call's other buffers on "
                                    f"{self.device}")
        want = _TORCH_DTYPES[dtype] if _TORCH_DTYPES else _torch_dtype(dtype)
        if t.dtype != want:
            raise FsdpArgumentError(f"{name} has dtype {t.dtype}, the layout needs {want}")
        if t.numel() < numel:
            raise FsdpArgumentError(f"{name} has {t.numel()} elements, the layout needs {numel}")
        if not t.is_contiguous():
            raise FsdpArgumentError(f"{name} is not contiguous")
        return t.data_ptr()

    def array(self, tensors, count: int, name: str, numel, dtype: int, allow_none=False):
        """C array of `count` pointers; `numel` is one int or one per entry."""
        if tensors is None:
            if allow_none:
                return None
            raise FsdpArgumentError(f"{name}: expected {count} tensors, got None")
        if len(tensors) != count:
            raise FsdpArgumentError(f"{name}: expected {count} tensors, got {len(tensors)}")
        arr = (_vp * max(1, count))()
        for k, t in enumerate(tensors):
            n = numel if isinstance(numel, int) else numel[k]
            arr[k] = self.one(t, f"{name}[{k}]", n, dtype)
        return arr


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return _vp(stream.cuda_stream)


def fsdp_pack_flat(layout: Layout, full, param_shard, master, stream=None) -> None:
    """Shard the full fp32 unit into every rank's master (and bf16) buffer."""
    R, P, S = layout.R, layout.full_numel, layout.shard_numel
    a = _Args()
    fp = _vp(a.one(full, "full", P, FSDP_F32))
    ps = a.array(param_shard, R, "param_shard", S, FSDP_BF16, allow_none=True)
    ms = a.array(master, R, "master", S, FSDP_F32)
    _check(load().fsdp_pack_flat(layout.handle, fp, ps, ms, _stream_handle(stream)))


def fsdp_all_gather_unflatten(layout: Layout, shard, full_out, stream=None) -> None:
    """Rebuild every destination rank's full unit from the R shard buffers."""
    R, pd = layout.R, layout.param_dtype
    a = _Args()
    fo = a.array(full_out, R, "full_out", layout.full_numel, pd)
    sh = a.array(shard, R, "shard", layout.shard_numel, pd)
    _check(load().fsdp_all_gather_unflatten(layout.handle, sh, fo, _stream_handle(stream)))


def _rs_arrays(a: _Args, R, P, S, grad_dtype, param_dtype, grad_full, master, m, v,
               param_shard_out, grad_shard_out):
    ma = a.array(master, R, "master", S, FSDP_F32)
    return (a.array(grad_full, R, "grad_full", P, grad_dtype), ma,
            a.array(m, R, "m", S, FSDP_F32), a.array(v, R, "v", S, FSDP_F32),
            a.array(param_shard_out, R, "param_shard_out", S, FSDP_BF16, allow_none=True),
            a.array(grad_shard_out, R, "grad_shard_out", S, FSDP_F32, allow_none=True))


def fsdp_reduce_scatter_adamw(layout: Layout, grad_full, master, m, v, param_shard_out,
                              grad_shard_out, hp: AdamWHP, step: int, stream=None) -> None:
    """Fixed-order fp32 reduce-scatter fused with the sharded AdamW step."""
    arrs = _rs_arrays(_Args(), layout.R, layout.full_numel, layout.shard_numel,
                      layout.grad_dtype, layout.param_dtype, grad_full, master, m, v,
                      param_shard_out, grad_shard_out)
    _check(load().fsdp_reduce_scatter_adamw(layout.handle, *arrs, ctypes.byref(hp), int(step),
                                            _stream_handle(stream)))


def fsdp_reduce_scatter_adamw_gather(layout: Layout, grad_full, master, m, v, param_shard_out,
                                     grad_shard_out, hp: AdamWHP, step: int,
                                     gather_layout: Layout, shard, full_out, stream=None) -> None:
    """Reduce-scatter + AdamW of one unit, then the all-gather of another (prefetch)."""
    a = _Args()
    arrs = _rs_arrays(a, layout.R, layout.full_numel, layout.shard_numel, layout.grad_dtype,
                      layout.param_dtype, grad_full, master, m, v, param_shard_out,
                      grad_shard_out)
    G, gd = gather_layout.R, gather_layout.param_dtype
    sh = a.array(shard, G, "shard", gather_layout.shard_numel, gd)
    fo = a.array(full_out, G, "full_out", gather_layout.full_numel, gd)
    _check(load().fsdp_reduce_scatter_adamw_gather(
        layout.handle, *arrs, ctypes.byref(hp), int(step), gather_layout.handle, sh, fo,
        _stream_handle(stream)))


def fsdp_adamw_from_reduced(layout: Layout, grad_avg_full, master, m, v, param_shard_out,
                            hp: AdamWHP, step: int, stream=None) -> None:
    """ZeRO-1's step: AdamW on each rank's own elements from its full,
    already averaged fp32 gradient (fsdp_all_reduce's fp32 output)."""
    R, P, S = layout.R, layout.full_numel, layout.shard_numel
    a = _Args()
    arrs = (a.array(grad_avg_full, R, "grad_avg_full", P, FSDP_F32),
            a.array(master, R, "master", S, FSDP_F32), a.array(m, R, "m", S, FSDP_F32),
            a.array(v, R, "v", S, FSDP_F32),
            a.array(param_shard_out, R, "param_shard_out", S, FSDP_BF16, allow_none=True))
    _check(load().fsdp_adamw_from_reduced(layout.handle, *arrs, ctypes.byref(hp), int(step),
                                          _stream_handle(stream)))


def fsdp_all_reduce(layout: Layout, grad_full, out, out_dtype: int, stream=None) -> None:
    """DDP all-reduce: every rank's output gets the fixed-order average."""
    R, P = layout.R, layout.full_numel
    a = _Args()
    if out_dtype not in (FSDP_F32, FSDP_BF16):
        raise FsdpArgumentError(f"out_dtype {out_dtype} is not FSDP_F32 or FSDP_BF16")
    o = a.array(out, R, "out", P, out_dtype)
    g = a.array(grad_full, R, "grad_full", P, layout.grad_dtype)
    _check(load().fsdp_all_reduce(layout.handle, g, o, int(out_dtype), _stream_handle(stream)))


def fsdp_accumulate_grad(layout: Layout, acc_full, grad_full, first: bool, stream=None) -> None:
    """Add one micro-batch's gradients into the R fp32 accumulators (copy if first)."""
    R, P = layout.R, layout.full_numel
    a = _Args()
    acc = a.array(acc_full, R, "acc_full", P, FSDP_F32)
    g = a.array(grad_full, R, "grad_full", P, layout.grad_dtype)
    _check(load().fsdp_accumulate_grad(layout.handle, acc, g, int(bool(first)),
                                       _stream_handle(stream)))


def fsdp_reduce_scatter_adamw_accum(layout: Layout, acc_full, grad_full, master, m, v,
                                    param_shard_out, grad_shard_out, hp: AdamWHP, step: int,
                                    stream=None) -> None:
    """The last micro-batch fused into reduce-scatter + AdamW."""
    a = _Args()
    arrs = _rs_arrays(a, layout.R, layout.full_numel, layout.shard_numel, layout.grad_dtype,
                      layout.param_dtype, grad_full, master, m, v, param_shard_out,
                      grad_shard_out)
    acc = a.array(acc_full, layout.R, "acc_full", layout.full_numel, FSDP_F32)
    _check(load().fsdp_reduce_scatter_adamw_accum(layout.handle, acc, *arrs, ctypes.byref(hp),
                                                  int(step), _stream_handle(stream)))


def _units_common(layouts):
    if not layouts:
        raise FsdpArgumentError("need at least one layout")
    lay = (_vp * len(layouts))(*[L.handle for L in layouts])
    R = layouts[0].R
    return lay, R


def _flat(per_unit, n_units, R, name):
    """Per-unit lists of R tensors, flattened unit-major (entry u*R + r)."""
    if per_unit is None:
        return None
    if len(per_unit) != n_units:
        raise FsdpArgumentError(f"{name}: expected {n_units} lists, got {len(per_unit)}")
    out = []
    for u, ts in enumerate(per_unit):
        if ts is None or len(ts) != R:
            raise FsdpArgumentError(f"{name}[{u}]: expected {R} tensors")
        out.extend(ts)
    return out


def fsdp_all_gather_unflatten_units(layouts, shard, full_out, stream=None) -> None:
    """All-gather + unflatten of several units in one launch. ``shard[u]`` and
    ``full_out[u]`` are unit u's lists of R tensors."""
    lay, R = _units_common(layouts)
    n = len(layouts)
    pd = layouts[0].param_dtype
    a = _Args()
    fo = a.array(_flat(full_out, n, R, "full_out"), n * R, "full_out",
                 [L.full_numel for L in layouts for _ in range(R)], pd)
    sh = a.array(_flat(shard, n, R, "shard"), n * R, "shard",
                 [L.shard_numel for L in layouts for _ in range(R)], pd)
    _check(load().fsdp_all_gather_unflatten_units(n, lay, sh, fo, _stream_handle(stream)))


def fsdp_reduce_scatter_adamw_units(layouts, grad_full, master, m, v, param_shard_out,
                                    grad_shard_out, hp: AdamWHP, step: int, stream=None) -> None:
    """Reduce-scatter + AdamW of several units in one launch; every argument
    but ``hp`` and ``step`` is a per-unit list of R tensors (or None)."""
    lay, R = _units_common(layouts)
    n = len(layouts)
    P = [L.full_numel for L in layouts for _ in range(R)]
    S = [L.shard_numel for L in layouts for _ in range(R)]
    a = _Args()
    ma = a.array(_flat(master, n, R, "master"), n * R, "master", S, FSDP_F32)
    g = a.array(_flat(grad_full, n, R, "grad_full"), n * R, "grad_full", P,
                layouts[0].grad_dtype)
    mm = a.array(_flat(m, n, R, "m"), n * R, "m", S, FSDP_F32)
    vv = a.array(_flat(v, n, R, "v"), n * R, "v", S, FSDP_F32)
    ps = a.array(_flat(param_shard_out, n, R, "param_shard_out"), n * R, "param_shard_out", S,
                 FSDP_BF16, allow_none=True)
    gs = a.array(_flat(grad_shard_out, n, R, "grad_shard_out"), n * R, "grad_shard_out", S,
                 FSDP_F32, allow_none=True)
    _check(load().fsdp_reduce_scatter_adamw_units(n, lay, g, ma, mm, vv, ps, gs,
                                                  ctypes.byref(hp), int(step),
                                                  _stream_handle(stream)))


# -- prepared calls ------------------------------------------------------------
#
# A training loop calls the same collectives on the same buffers every step.
# A prepared call checks and marshals its tensors once; each later call is one
# C call with the step's scalars, which matters for small units, where the
# per-tensor checks above cost more host time than the kernels take on the
# GPU. The prepared call holds references to its tensors, so they stay
# allocated while it lives; the C library still validates every call.

class PreparedCall:
    """One library call with its tensor arguments bound."""

    def __init__(self, fn, head, arrays, tensors, takes_step: bool):
        self._fn, self._head, self._arrays = fn, head, arrays
        self._tensors = tensors  # keeps the buffers alive
        self._takes_step = takes_step
        self._stream_cache = (None, None)

    def _stream(self, stream):
        if stream is None:
            return _stream_handle(None)
        key, handle = self._stream_cache
        if key is not stream:
            handle = _vp(stream.cuda_stream)
            self._stream_cache = (stream, handle)
        return handle

    def __call__(self, hp: AdamWHP | None = None, step: int | None = None, stream=None) -> None:
        if self._takes_step:
            if hp is None or step is None:
                raise FsdpArgumentError("this call needs hp and step")
            _check(self._fn(*self._head, *self._arrays, ctypes.byref(hp), int(step),
                            self._stream(stream)))
        else:
            _check(self._fn(*self._head, *self._arrays, self._stream(stream)))


def prepare_fsdp_all_gather_unflatten(layout: Layout, shard, full_out) -> PreparedCall:
    R, pd = layout.R, layout.param_dtype
    a = _Args()
    fo = a.array(full_out, R, "full_out", layout.full_numel, pd)
    sh = a.array(shard, R, "shard", layout.shard_numel, pd)
    return PreparedCall(load().fsdp_all_gather_unflatten, (layout.handle,), (sh, fo),
                        (layout, list(shard), list(full_out)), False)


def prepare_fsdp_reduce_scatter_adamw(layout: Layout, grad_full, master, m, v, param_shard_out,
                                 grad_shard_out=None) -> PreparedCall:
    arrs = _rs_arrays(_Args(), layout.R, layout.full_numel, layout.shard_numel,
                      layout.grad_dtype, layout.param_dtype, grad_full, master, m, v,
                      param_shard_out, grad_shard_out)
    return PreparedCall(load().fsdp_reduce_scatter_adamw, (layout.handle,), arrs,
                        (layout, grad_full, master, m, v, param_shard_out, grad_shard_out), True)


def prepare_fsdp_all_gather_unflatten_units(layouts, shard, full_out) -> PreparedCall:
    lay, R = _units_common(layouts)
    n = len(layouts)
    pd = layouts[0].param_dtype
    a = _Args()
    fo = a.array(_flat(full_out, n, R, "full_out"), n * R, "full_out",
                 [L.full_numel for L in layouts for _ in range(R)], pd)
    sh = a.array(_flat(shard, n, R, "shard"), n * R, "shard",
                 [L.shard_numel for L in layouts for _ in range(R)], pd)
    return PreparedCall(load().fsdp_all_gather_unflatten_units, (n, lay), (sh, fo),
                        (list(layouts), shard, full_out), False)


def prepare_fsdp_reduce_scatter_adamw_units(layouts, grad_full, master, m, v, param_shard_out,
                                       grad_shard_out=None) -> PreparedCall:
    lay, R = _units_common(layouts)
    n = len(layouts)
    P = [L.full_numel for L in layouts for _ in range(R)]
    S = [L.shard_numel for L in layouts for _ in range(R)]
    a = _Args()
    ma = a.array(_flat(master, n, R, "master"), n * R, "master", S, FSDP_F32)
    g = a.array(_flat(grad_full, n, R, "grad_full"), n * R, "grad_full", P,
                layouts[0].grad_dtype)
    mm = a.array(_flat(m, n, R, "m"), n * R, "m", S, FSDP_F32)
    vv = a.array(_flat(v, n, R, "v"), n * R, "v", S, FSDP_F32)
    ps = a.array(_flat(param_shard_out, n, R, "param_shard_out"), n * R, "param_shard_out", S,
                 FSDP_BF16, allow_none=True)
    gs = a.array(_flat(grad_shard_out, n, R, "grad_shard_out"), n * R, "grad_shard_out", S,
                 FSDP_F32, allow_none=True)
    return PreparedCall(load().fsdp_reduce_scatter_adamw_units, (n, lay),
                        (g, ma, mm, vv, ps, gs),
                        (list(layouts), grad_full, master, m, v, param_shard_out,
                         grad_shard_out), True)


def fsdp_write_stream(dst, pattern: int = 0x3FC03FC0, stream=None) -> None:
    """Measurement helper: write a 32-bit pattern over every tensor in
    ``dst`` (equal sizes, a multiple of 32 bytes) with the all-gather's store
    pattern, to time the write-only stream ceiling."""
    if not dst:
        raise FsdpArgumentError("dst: need at least one tensor")
    nbytes = dst[0].numel() * dst[0].element_size()
    a = _Args()
    arr = a.array(dst, len(dst), "dst", dst[0].numel(), FSDP_BF16 if dst[0].element_size() == 2
                  else FSDP_F32)
    _check(load().fsdp_write_stream(arr, len(dst), nbytes, pattern & 0xFFFFFFFF,
                                    _stream_handle(stream)))


def fsdp_stage_wait_timeouts(device=None) -> int:
    """Thread blocks of the staged reduce-scatter on ``device`` (default:
    the current CUDA device) that gave up waiting for their gradient copies
    since the library was loaded; 0 in every valid run. Synchronises the
    device."""
    n = ctypes.c_uint64(0)
    _check(load().fsdp_stage_wait_timeouts(_device_index(device), ctypes.byref(n)))
    return int(n.value)


def _device_index(device) -> int:
    import torch
    d = torch.device("cuda", device) if isinstance(device, int) else \
        torch.device(device if device is not None else "cuda")
    return d.index if d.index is not None else torch.cuda.current_device()


def fsdp_stage_wait_selftest(device=None) -> int:
    """One thread block waits on an mbarrier that nothing completes, gives up
    after 20 ms and counts itself; returns that count (1)."""
    n = ctypes.c_uint64(0)
    _check(load().fsdp_stage_wait_selftest(_device_index(device), ctypes.byref(n)))
    return int(n.value)


def fsdp_version() -> str:
    return load().fsdp_version().decode()
