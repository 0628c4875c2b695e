"""CPU oracle of the FSDP per-unit shard engine.

TEST INFRASTRUCTURE. This package is the checker the CUDA path is compared
against; it shares no code with that path. Only ``tests/``, the smoke check in
``__graft_entry__`` and the benchmark's CPU-baseline / reference leg may import
it. The product path never routes through it.

``fsdp_oracle.c`` holds the arithmetic (plain scalar C, IEEE binary32 with no
contraction); this module only marshals numpy arrays into it. ``brute.py``
is an independent pure-Python restatement for tiny integer cases and
``formulas.py`` holds the pages' memory and communication formulas.

bf16 values are carried as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

FLAT = 1        # FSDP1 FlatParameter
PER_PARAM = 2   # FSDP2 per-parameter Shard(0)
ZERO3 = 3       # ZeRO-3 inter-tensor: whole tensors on owner ranks
F32 = 0
BF16 = 1
SEG_ALIGN = 8   # per-parameter shard segments are padded to a multiple of 8 elements

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fsdp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libfsdp_oracle.so")
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)
_vpp = ctypes.POINTER(ctypes.c_void_p)


_OMP_LIB_PATH = os.path.join(_HERE, "libfsdp_oracle_omp.so")


def build(force: bool = False, openmp: bool = False) -> str:
    """Compile the C oracle into ``oracle/libfsdp_oracle.so`` (gcc, no
    contraction), or with ``openmp`` the same source with -fopenmp into
    ``oracle/libfsdp_oracle_omp.so`` (element loops split over threads,
    per-element arithmetic unchanged)."""
    path = _OMP_LIB_PATH if openmp else _LIB_PATH
    if (not force and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           *(["-fopenmp"] if openmp else []), "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def _load(path: str):
    L = ctypes.CDLL(path)
    L.orc_rank_rows.restype = ctypes.c_int64
    L.orc_rank_rows.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _i64p]
    L.orc_layout.restype = ctypes.c_int
    L.orc_layout.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _i64p, _i64p,
                             _i64p, _i64p, _i64p, _i64p]
    L.orc_f32_to_bf16.restype = ctypes.c_uint16
    L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
    L.orc_bf16_to_f32.restype = ctypes.c_float
    L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_f32_to_bf16_array.restype = None
    L.orc_f32_to_bf16_array.argtypes = [ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    L.orc_pack.restype = ctypes.c_int
    L.orc_pack.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _i64p, _i64p,
                           ctypes.c_void_p, _vpp, _vpp]
    L.orc_all_gather.restype = ctypes.c_int
    L.orc_all_gather.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _i64p, _i64p,
                                 ctypes.c_int64, _vpp, _vpp]
    L.orc_sum_ranks.restype = None
    L.orc_sum_ranks.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _vpp,
                                ctypes.c_void_p]
    L.orc_reduce_scatter.restype = ctypes.c_int
    L.orc_reduce_scatter.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _i64p,
                                     _i64p, ctypes.c_int, _vpp, _vpp]
    L.orc_adamw.restype = None
    L.orc_adamw.argtypes = [ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                            ctypes.c_void_p, ctypes.c_void_p,
                            ctypes.POINTER(ctypes.c_double), ctypes.c_int64]
    L.orc_zero3_owners.restype = ctypes.c_int
    L.orc_zero3_owners.argtypes = [ctypes.c_int64, ctypes.c_int64, _i64p, _i64p, _i64p]
    L.orc_owner.restype = ctypes.c_int
    L.orc_owner.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _i64p, _i64p,
                            ctypes.c_int64, _i64p, _i64p, _i64p]
    L.orc_all_reduce.restype = None
    L.orc_all_reduce.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _vpp,
                                 ctypes.c_int, _vpp]
    L.orc_accumulate.restype = None
    L.orc_accumulate.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _vpp, _vpp,
                                 ctypes.c_int]
    L.orc_rs_adamw.restype = ctypes.c_int
    L.orc_rs_adamw.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _i64p, _i64p,
                               ctypes.c_int, _vpp, _vpp, _vpp, _vpp, _vpp, _vpp,
                               ctypes.POINTER(ctypes.c_double), ctypes.c_int64]
    return L


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = _load(_LIB_PATH)
    return _lib


def use_library(path: str) -> None:
    """Point this module at another build of the oracle source for the rest of
    the process: a copy with a planted mistake (the tests that check the pins
    catch it), or the OpenMP build (the timed CPU baseline)."""
    global _lib
    _lib = _load(path)


class using:
    """Context manager: the oracle functions use the library at ``path``
    inside the block and the plain build after it."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        use_library(self.path)
        return self

    def __exit__(self, *exc):
        use_library(build())


def _i64(values) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(values, dtype=np.int64))


def _p(a: np.ndarray):
    return ctypes.cast(a.ctypes.data, _i64p)


def _ptrs(arrays) -> ctypes.Array:
    out = (ctypes.c_void_p * max(1, len(arrays)))()
    for k, a in enumerate(arrays):
        if a is not None:
            assert a.flags["C_CONTIGUOUS"]
            out[k] = a.ctypes.data
    return out


def _dims(shapes):
    d0, inner = [], []
    for shp in shapes:
        shp = tuple(int(x) for x in shp)
        d0.append(shp[0] if len(shp) else 1)
        inner.append(int(np.prod(shp[1:], dtype=np.int64)) if len(shp) > 1 else 1)
    return _i64(d0), _i64(inner)


@dataclass
class Layout:
    """The oracle's view of one FSDP unit's layout."""
    mode: int
    R: int
    shapes: list
    d0: np.ndarray
    inner: np.ndarray
    full_off: np.ndarray     # per parameter, offset in the full unit
    shard_off: np.ndarray    # per parameter, offset in a rank's shard buffer (PER_PARAM)
    shard_rows: np.ndarray   # per parameter, s_i = ceil(d0_i / R)
    full_numel: int          # P
    shard_numel: int         # per-rank shard buffer length (with padding)
    padded_numel: int        # FLAT: R * S
    owner: np.ndarray = None  # ZERO3: owner rank of every parameter

    def rank_rows(self, i: int, r: int):
        """(first row, row count) of parameter i held by rank r."""
        if self.mode == ZERO3:
            return 0, (int(self.d0[i]) if int(self.owner[i]) == r else 0)
        start = ctypes.c_int64(0)
        cnt = lib().orc_rank_rows(int(self.d0[i]), self.R, r, ctypes.byref(start))
        return int(start.value), int(cnt)

    def rank_numel(self, r: int) -> int:
        """Number of real (non-padding) elements rank r owns."""
        if self.mode == FLAT:
            j = r * self.shard_numel
            return max(0, min(self.shard_numel, self.full_numel - j))
        return sum(self.rank_rows(i, r)[1] * int(self.inner[i]) for i in range(len(self.shapes)))


def layout(mode: int, R: int, shapes) -> Layout:
    d0, inner = _dims(shapes)
    n = len(d0)
    full_off = np.zeros(max(1, n), np.int64)
    shard_off = np.zeros(max(1, n), np.int64)
    rows = np.zeros(max(1, n), np.int64)
    out = np.zeros(3, np.int64)
    rc = lib().orc_layout(mode, R, n, _p(d0 if n else _i64([0])), _p(inner if n else _i64([0])),
                          _p(full_off), _p(shard_off), _p(rows), _p(out))
    if rc != 0:
        raise ValueError("oracle: bad layout arguments")
    owner = None
    if mode == ZERO3:
        owner = np.zeros(max(1, n), np.int64)
        lib().orc_zero3_owners(R, n, _p(d0 if n else _i64([0])), _p(inner if n else _i64([0])),
                               _p(owner))
        owner = owner[:n]
    return Layout(mode, R, [tuple(s) for s in shapes], d0, inner, full_off[:n], shard_off[:n],
                  rows[:n], int(out[0]), int(out[1]), int(out[2]), owner)


def f32_to_bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    y = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_bf16_array(x.size, x.ctypes.data, y.ctypes.data)
    return y


def bf16_to_f32(h) -> np.ndarray:
    """Exact widening (bf16 is the upper half of a binary32)."""
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << np.uint32(16)).view(np.float32)


def pack(L: Layout, full_f32: np.ndarray, with_bf16: bool):
    """Shard buffers from the full fp32 unit: (masters, bf16 copies or None)."""
    full_f32 = np.ascontiguousarray(full_f32, dtype=np.float32)
    assert full_f32.size == L.full_numel
    masters = [np.zeros(L.shard_numel, np.float32) for _ in range(L.R)]
    p16 = [np.zeros(L.shard_numel, np.uint16) for _ in range(L.R)] if with_bf16 else None
    rc = lib().orc_pack(L.mode, L.R, len(L.d0), _p(L.d0), _p(L.inner), full_f32.ctypes.data,
                        _ptrs(masters), _ptrs(p16) if p16 else _ptrs([None] * L.R))
    assert rc == 0
    return masters, p16


def all_gather(L: Layout, shards) -> list:
    """R full units (one per destination rank) from the R shard buffers."""
    assert len(shards) == L.R
    dt = shards[0].dtype
    shards = [np.ascontiguousarray(s) for s in shards]
    full = [np.zeros(L.full_numel, dt) for _ in range(L.R)]
    rc = lib().orc_all_gather(L.mode, L.R, len(L.d0), _p(L.d0), _p(L.inner), dt.itemsize,
                              _ptrs(shards), _ptrs(full))
    assert rc == 0
    return full


def _gdtype(g) -> int:
    return BF16 if g.dtype == np.uint16 else F32


def sum_ranks(grads_at) -> np.ndarray:
    """Fixed-order fp32 sum over ranks of matching elements, times fl(1/R).

    ``grads_at[q]`` holds rank q's values (uint16 = bf16 bits, or float32)."""
    R = len(grads_at)
    g = [np.ascontiguousarray(x) for x in grads_at]
    out = np.empty(g[0].size, np.float32)
    lib().orc_sum_ranks(R, g[0].size, _gdtype(g[0]), _ptrs(g), out.ctypes.data)
    return out


def reduce_scatter(L: Layout, grads) -> list:
    """Per-rank fp32 gradient shards (shard-buffer layout, zero padding)."""
    assert len(grads) == L.R
    grads = [np.ascontiguousarray(g) for g in grads]
    out = [np.zeros(L.shard_numel, np.float32) for _ in range(L.R)]
    rc = lib().orc_reduce_scatter(L.mode, L.R, len(L.d0), _p(L.d0), _p(L.inner),
                                  _gdtype(grads[0]), _ptrs(grads), _ptrs(out))
    assert rc == 0
    return out


@dataclass
class AdamWHP:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01

    def as_c(self):
        return (ctypes.c_double * 5)(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay)


def adamw(g, w, m, v, hp: AdamWHP, t: int) -> None:
    """In-place AdamW step on contiguous float32 arrays of equal length."""
    for a in (g, w, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    lib().orc_adamw(w.size, g.ctypes.data, w.ctypes.data, m.ctypes.data, v.ctypes.data,
                    hp.as_c(), int(t))


def rs_adamw(L: Layout, grads, master, m, v, hp: AdamWHP, t: int, with_bf16: bool):
    """Reduce-scatter + sharded AdamW, in place on master/m/v.

    Returns (fp32 gradient shards, bf16 parameter shards or None)."""
    grads = [np.ascontiguousarray(g) for g in grads]
    gsh = [np.zeros(L.shard_numel, np.float32) for _ in range(L.R)]
    p16 = [np.zeros(L.shard_numel, np.uint16) for _ in range(L.R)] if with_bf16 else None
    rc = lib().orc_rs_adamw(L.mode, L.R, len(L.d0), _p(L.d0), _p(L.inner), _gdtype(grads[0]),
                            _ptrs(grads), _ptrs(master), _ptrs(m), _ptrs(v), _ptrs(gsh),
                            _ptrs(p16) if p16 else _ptrs([None] * L.R), hp.as_c(), int(t))
    assert rc == 0
    return gsh, p16


def owner(L: Layout, js) -> tuple:
    """(rank, shard-buffer index) holding each unit element index in ``js``."""
    js = _i64(js).ravel()
    rank = np.zeros(js.size, np.int64)
    index = np.zeros(js.size, np.int64)
    rc = lib().orc_owner(L.mode, L.R, len(L.d0), _p(L.d0), _p(L.inner), js.size, _p(js),
                         _p(rank), _p(index))
    if rc != 0:
        raise ValueError("oracle: element index outside the unit")
    return rank, index


def all_reduce(grads, out_bf16: bool) -> list:
    """DDP all-reduce: R identical full outputs of the fixed-order average
    (float32, or bf16 bits as uint16)."""
    grads = [np.ascontiguousarray(g) for g in grads]
    R, P = len(grads), grads[0].size
    dt = np.uint16 if out_bf16 else np.float32
    out = [np.zeros(P, dt) for _ in range(R)]
    lib().orc_all_reduce(R, P, _gdtype(grads[0]), _ptrs(grads), BF16 if out_bf16 else F32,
                         _ptrs(out))
    return out


def accumulate(acc, grads, first: bool) -> None:
    """In place: acc[q] = g[q] (first micro-batch) or acc[q] + g[q], fp32."""
    grads = [np.ascontiguousarray(g) for g in grads]
    for a in acc:
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    lib().orc_accumulate(len(grads), grads[0].size, _gdtype(grads[0]), _ptrs(acc),
                         _ptrs(grads), int(bool(first)))
