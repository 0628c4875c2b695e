"""The C-ABI library on the host (no GPU): it loads, exports every symbol the
header declares, its layout agrees with the oracle's, and every argument
error is caught on the host before any CUDA call."""
import ctypes
import re
from pathlib import Path

import numpy as np
import pytest

import oracle
from fully_sharded_state_gb300 import build, capi
from fully_sharded_state_gb300.synth import WORKLOADS

HEADER_DIR = Path(__file__).resolve().parent.parent / "include"


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi.load()


def declared_functions():
    names = set()
    for h in HEADER_DIR.glob("*.h"):
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ ]*?[\s\*]+"
                                r"(fsdp_[A-Za-z0-9_]+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fsdp_layout", "fsdp_pack_flat", "fsdp_all_gather_unflatten",
              "fsdp_reduce_scatter_adamw", "fsdp_layout_query", "fsdp_layout_destroy",
              "fsdp_last_error", "fsdp_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert b"sm_103a" in lib.fsdp_version()


_OMODE = {capi.FSDP_FLAT: oracle.FLAT, capi.FSDP_PER_PARAM: oracle.PER_PARAM,
          capi.FSDP_ZERO3: oracle.ZERO3}


def _both_layouts(mode, R, shapes, pdt=capi.FSDP_BF16, gdt=capi.FSDP_BF16):
    L = capi.fsdp_layout(mode, R, shapes, pdt, gdt)
    O = oracle.layout(_OMODE[mode], R, shapes)
    return L, O


def _compare(L, O):
    assert L.full_numel == O.full_numel
    assert L.shard_numel == O.shard_numel
    assert L.query(capi.Q_PADDED_NUMEL) == L.R * O.shard_numel
    for i in range(len(O.shapes)):
        assert L.param_full_offset(i) == O.full_off[i]
        assert L.query(capi.Q_PARAM_SHARD_ROWS, i) == O.shard_rows[i]
        if O.mode != oracle.FLAT:
            assert L.param_shard_offset(i) == O.shard_off[i]
        if O.mode == oracle.ZERO3:
            assert L.param_owner(i) == O.owner[i]
        for r in range(L.R):
            s, c = O.rank_rows(i, r)
            got = L.rank_rows(i, r)
            assert got[1] == c and (c == 0 or got[0] == s)
    for r in range(L.R):
        assert L.rank_numel(r) == O.rank_numel(r)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_layout_matches_oracle_on_workloads(lib, name):
    wl = WORKLOADS[name]
    mode = capi.FSDP_FLAT if wl.mode == "flat" else capi.FSDP_PER_PARAM
    for u in range(len(wl.units)):
        _compare(*_both_layouts(mode, wl.R, wl.unit_shapes(u)))
        _compare(*_both_layouts(capi.FSDP_ZERO3, wl.R, wl.unit_shapes(u)))


def test_layout_matches_oracle_random(lib):
    rng = np.random.default_rng(21)
    for trial in range(300):
        n = int(rng.integers(0, 12))
        shapes = []
        for _ in range(n):
            nd = int(rng.integers(1, 4))
            shapes.append(tuple([int(rng.integers(0, 300))] +
                                [int(rng.integers(1, 70)) for _ in range(nd - 1)]))
        R = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 16, 33, 64]))
        for mode in (capi.FSDP_PER_PARAM, capi.FSDP_FLAT, capi.FSDP_ZERO3):
            _compare(*_both_layouts(mode, R, shapes))


def test_layout_many_params_spans_several_launch_plans(lib):
    shapes = [(k % 7 + 1, 3) for k in range(1000)]
    _compare(*_both_layouts(capi.FSDP_PER_PARAM, 8, shapes))
    _compare(*_both_layouts(capi.FSDP_ZERO3, 8, shapes))


def test_owner_query_only_for_zero3(lib):
    L = capi.fsdp_layout(capi.FSDP_PER_PARAM, 4, [(8, 2)], capi.FSDP_BF16, capi.FSDP_BF16)
    out = ctypes.c_int64()
    assert lib.fsdp_layout_query(L.handle, capi.Q_PARAM_OWNER, 0, 0, ctypes.byref(out)) == \
        capi.FSDP_EINVAL


# ------------------------------------------------------------------ errors --

def _raw_layout(lib, mode=capi.FSDP_PER_PARAM, R=2, dims=((4, 1),), pdt=capi.FSDP_BF16,
                gdt=capi.FSDP_BF16):
    n = len(dims)
    d0 = (ctypes.c_int64 * max(1, n))(*[d[0] for d in dims])
    inner = (ctypes.c_int64 * max(1, n))(*[d[1] for d in dims])
    h = ctypes.c_void_p()
    st = lib.fsdp_layout(mode, R, n, d0, inner, pdt, gdt, ctypes.byref(h))
    return st, h


@pytest.mark.parametrize("kw,status", [
    (dict(R=0), capi.FSDP_EINVAL),
    (dict(R=65), capi.FSDP_EINVAL),
    (dict(mode=4), capi.FSDP_EINVAL),
    (dict(dims=((-1, 4),)), capi.FSDP_EINVAL),
    (dict(dims=((4, -2),)), capi.FSDP_EINVAL),
    (dict(dims=((1 << 40, 1 << 30),)), capi.FSDP_ERANGE),
    (dict(dims=((1 << 61, 1), (1 << 61, 1))), capi.FSDP_ERANGE),
    (dict(pdt=7), capi.FSDP_EUNSUPPORTED),
    (dict(gdt=2), capi.FSDP_EUNSUPPORTED),
])
def test_layout_rejects_bad_arguments(lib, kw, status):
    st, h = _raw_layout(lib, **kw)
    assert st == status
    assert not h.value
    assert lib.fsdp_last_error()


def test_layout_accepts_empty_units_and_params(lib):
    for dims in ((), ((0, 5),), ((3, 0),), ((0, 0), (1, 1))):
        st, h = _raw_layout(lib, dims=dims)
        assert st == capi.FSDP_OK
        lib.fsdp_layout_destroy(h)
    assert lib.fsdp_layout(capi.FSDP_PER_PARAM, 2, 1, None, None, 0, 0,
                           ctypes.byref(ctypes.c_void_p())) == capi.FSDP_EINVAL
    assert lib.fsdp_layout(capi.FSDP_PER_PARAM, 2, 0, None, None, 0, 0, None) == capi.FSDP_EINVAL


def test_query_rejects_bad_indices(lib):
    L = capi.fsdp_layout(capi.FSDP_FLAT, 4, [(8, 2)], capi.FSDP_BF16, capi.FSDP_BF16)
    out = ctypes.c_int64()
    for what, i, r in ((capi.Q_PARAM_FULL_OFFSET, 1, 0), (capi.Q_PARAM_RANK_ROWS, 0, 4),
                       (capi.Q_RANK_NUMEL, 0, -1), (capi.Q_PARAM_SHARD_OFFSET, 0, 0), (99, 0, 0)):
        assert lib.fsdp_layout_query(L.handle, what, i, r, ctypes.byref(out)) == capi.FSDP_EINVAL
    assert lib.fsdp_layout_query(None, capi.Q_FULL_NUMEL, 0, 0, ctypes.byref(out)) == \
        capi.FSDP_EINVAL


def _ptrs(values):
    arr = (ctypes.c_void_p * len(values))()
    for k, x in enumerate(values):
        arr[k] = x
    return arr


BASE = 0x7f0000000000  # fake, never dereferenced: validation fails first


def _hp(**kw):
    d = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    d.update(kw)
    return capi.AdamWHP(**d)


def _rs_args(R=2, P_bytes=1 << 20, **over):
    a = dict(grad=_ptrs([BASE + k * P_bytes for k in range(R)]),
             master=_ptrs([BASE + (10 + k) * P_bytes for k in range(R)]),
             m=_ptrs([BASE + (20 + k) * P_bytes for k in range(R)]),
             v=_ptrs([BASE + (30 + k) * P_bytes for k in range(R)]),
             pshard=_ptrs([BASE + (40 + k) * P_bytes for k in range(R)]),
             gshard=None, hp=_hp(), step=1)
    a.update(over)
    return a


def _call_rs(lib, L, a):
    return lib.fsdp_reduce_scatter_adamw(L.handle, a["grad"], a["master"], a["m"], a["v"],
                                         a["pshard"], a["gshard"], ctypes.byref(a["hp"]),
                                         a["step"], None)


@pytest.mark.parametrize("over,status", [
    (dict(step=0), capi.FSDP_EINVAL),
    (dict(hp=_hp(beta1=1.0)), capi.FSDP_EINVAL),
    (dict(hp=_hp(beta2=-0.1)), capi.FSDP_EINVAL),
    (dict(hp=_hp(eps=0.0)), capi.FSDP_EINVAL),
    (dict(hp=_hp(lr=float("nan"))), capi.FSDP_EINVAL),
    (dict(grad=None), capi.FSDP_EINVAL),
    (dict(grad=_ptrs([BASE, 0])), capi.FSDP_EINVAL),
    (dict(master=_ptrs([BASE + 10 * (1 << 20) + 4, BASE + 11 * (1 << 20)])), capi.FSDP_EALIGN),
    (dict(pshard=None), capi.FSDP_EINVAL),
    # master[1] overlaps m[0]
    (dict(master=_ptrs([BASE + 10 * (1 << 20), BASE + 20 * (1 << 20) + 64])), capi.FSDP_EINVAL),
    # gshard overlaps a gradient (an input)
    (dict(gshard=_ptrs([BASE + 64, BASE + 50 * (1 << 20)])), capi.FSDP_EINVAL),
])
def test_reduce_scatter_adamw_rejects_bad_arguments(lib, over, status):
    L = capi.fsdp_layout(capi.FSDP_PER_PARAM, 2, [(4096, 16)], capi.FSDP_BF16, capi.FSDP_BF16)
    assert _call_rs(lib, L, _rs_args(**over)) == status
    assert lib.fsdp_last_error()


def _call_adamw_reduced(lib, L, a):
    return lib.fsdp_adamw_from_reduced(L.handle if L else None, a["grad"], a["master"], a["m"],
                                       a["v"], a["pshard"], ctypes.byref(a["hp"]), a["step"],
                                       None)


@pytest.mark.parametrize("over,status", [
    (dict(step=0), capi.FSDP_EINVAL),
    (dict(hp=_hp(beta1=1.0)), capi.FSDP_EINVAL),
    (dict(grad=None), capi.FSDP_EINVAL),
    (dict(grad=_ptrs([BASE, 0])), capi.FSDP_EINVAL),
    (dict(master=_ptrs([BASE + 10 * (1 << 20) + 4, BASE + 11 * (1 << 20)])), capi.FSDP_EALIGN),
    (dict(pshard=None), capi.FSDP_EINVAL),
    # master[1] overlaps m[0]
    (dict(master=_ptrs([BASE + 10 * (1 << 20), BASE + 20 * (1 << 20) + 64])), capi.FSDP_EINVAL),
    # v[0] overlaps an averaged gradient (an input)
    (dict(v=_ptrs([BASE + 64, BASE + 31 * (1 << 20)])), capi.FSDP_EINVAL),
])
def test_adamw_from_reduced_rejects_bad_arguments(lib, over, status):
    L = capi.fsdp_layout(capi.FSDP_PER_PARAM, 2, [(4096, 16)], capi.FSDP_BF16, capi.FSDP_BF16)
    assert _call_adamw_reduced(lib, L, _rs_args(**over)) == status
    assert lib.fsdp_last_error()
    assert _call_adamw_reduced(lib, None, _rs_args()) == capi.FSDP_EINVAL


def test_f32_layouts_take_no_bf16_shard(lib):
    L = capi.fsdp_layout(capi.FSDP_PER_PARAM, 2, [(4096, 16)], capi.FSDP_F32, capi.FSDP_F32)
    assert _call_rs(lib, L, _rs_args()) == capi.FSDP_EINVAL
    full = ctypes.c_void_p(BASE)
    assert lib.fsdp_pack_flat(L.handle, full, _ptrs([BASE + 1 << 24, BASE + 2 << 24]),
                              _ptrs([BASE + 3 << 24, BASE + 4 << 24]), None) == capi.FSDP_EINVAL


def test_gather_and_pack_reject_bad_arguments(lib):
    L = capi.fsdp_layout(capi.FSDP_FLAT, 2, [(4096, 16)], capi.FSDP_BF16, capi.FSDP_BF16)
    MB = 1 << 20
    shard = _ptrs([BASE, BASE + MB])
    assert lib.fsdp_all_gather_unflatten(None, shard, shard, None) == capi.FSDP_EINVAL
    assert lib.fsdp_all_gather_unflatten(L.handle, shard, None, None) == capi.FSDP_EINVAL
    # destinations overlapping the sources
    assert lib.fsdp_all_gather_unflatten(L.handle, shard, _ptrs([BASE + 64, BASE + 4 * MB]),
                                         None) == capi.FSDP_EINVAL
    # two destinations overlapping each other
    assert lib.fsdp_all_gather_unflatten(L.handle, shard, _ptrs([BASE + 4 * MB, BASE + 4 * MB]),
                                         None) == capi.FSDP_EINVAL
    assert lib.fsdp_all_gather_unflatten(L.handle, shard, _ptrs([BASE + 4 * MB + 2,
                                                                 BASE + 8 * MB]),
                                         None) == capi.FSDP_EALIGN
    assert lib.fsdp_pack_flat(L.handle, None, _ptrs([BASE, BASE + MB]),
                              _ptrs([BASE + 2 * MB, BASE + 3 * MB]), None) == capi.FSDP_EINVAL
    assert lib.fsdp_pack_flat(L.handle, ctypes.c_void_p(BASE + 8 * MB), None,
                              _ptrs([BASE + 2 * MB, BASE + 3 * MB]), None) == capi.FSDP_EINVAL


def test_empty_unit_calls_are_no_ops(lib):
    L = capi.fsdp_layout(capi.FSDP_PER_PARAM, 4, [(0, 8)], capi.FSDP_BF16, capi.FSDP_BF16)
    nul = _ptrs([0, 0, 0, 0])
    assert lib.fsdp_all_gather_unflatten(L.handle, nul, nul, None) == capi.FSDP_OK
    assert _call_rs(lib, L, dict(grad=nul, master=nul, m=nul, v=nul, pshard=nul, gshard=None,
                                 hp=_hp(), step=1)) == capi.FSDP_OK


def test_binding_rejects_host_tensors(lib):
    torch = pytest.importorskip("torch")
    L = capi.fsdp_layout(capi.FSDP_PER_PARAM, 2, [(8,)], capi.FSDP_F32, capi.FSDP_F32)
    t = [torch.zeros(8), torch.zeros(8)]
    with pytest.raises(ValueError):
        capi.fsdp_all_gather_unflatten(L, t, t)


def test_all_reduce_rejects_bad_arguments(lib):
    L = capi.fsdp_layout(capi.FSDP_PER_PARAM, 2, [(4096, 16)], capi.FSDP_BF16, capi.FSDP_BF16)
    MB = 1 << 20
    g = _ptrs([BASE, BASE + MB])
    assert lib.fsdp_all_reduce(L.handle, g, _ptrs([BASE + 4 * MB, BASE + 8 * MB]), 7,
                               None) == capi.FSDP_EUNSUPPORTED
    # an output overlapping a gradient
    assert lib.fsdp_all_reduce(L.handle, g, _ptrs([BASE + 64, BASE + 8 * MB]), capi.FSDP_F32,
                               None) == capi.FSDP_EINVAL
    # fp32 outputs of 256 KB each overlap when placed 128 KB apart
    assert lib.fsdp_all_reduce(L.handle, g, _ptrs([BASE + 4 * MB, BASE + 4 * MB + (1 << 17)]),
                               capi.FSDP_F32, None) == capi.FSDP_EINVAL
    assert lib.fsdp_all_reduce(None, g, g, capi.FSDP_F32, None) == capi.FSDP_EINVAL


def test_accumulation_rejects_bad_arguments(lib):
    L = capi.fsdp_layout(capi.FSDP_PER_PARAM, 2, [(4096, 16)], capi.FSDP_BF16, capi.FSDP_BF16)
    MB = 1 << 20
    g = _ptrs([BASE, BASE + MB])
    acc = _ptrs([BASE + 4 * MB, BASE + 8 * MB])
    assert lib.fsdp_accumulate_grad(None, acc, g, 1, None) == capi.FSDP_EINVAL
    assert lib.fsdp_accumulate_grad(L.handle, _ptrs([BASE + 4 * MB + 8, BASE + 8 * MB]), g, 0,
                                    None) == capi.FSDP_EALIGN
    # an accumulator overlapping a gradient
    assert lib.fsdp_accumulate_grad(L.handle, _ptrs([BASE + 64, BASE + 8 * MB]), g, 0,
                                    None) == capi.FSDP_EINVAL
    a = _rs_args()
    # accumulators overlapping the master (an output)
    st = lib.fsdp_reduce_scatter_adamw_accum(L.handle, a["master"], a["grad"], a["master"],
                                             a["m"], a["v"], a["pshard"], None,
                                             ctypes.byref(a["hp"]), 1, None)
    assert st == capi.FSDP_EINVAL
    st = lib.fsdp_reduce_scatter_adamw_accum(L.handle, None, a["grad"], a["master"], a["m"],
                                             a["v"], a["pshard"], None, ctypes.byref(a["hp"]),
                                             1, None)
    assert st == capi.FSDP_EINVAL
    st = lib.fsdp_reduce_scatter_adamw_accum(L.handle, acc, a["grad"], a["master"], a["m"],
                                             a["v"], a["pshard"], None, ctypes.byref(a["hp"]),
                                             0, None)
    assert st == capi.FSDP_EINVAL


# ---- the binding's checks of tensor arguments (tensor metadata only) -------

class FakeTensor:
    """Metadata of a CUDA tensor, enough for the binding's checks; its data
    pointer is never dereferenced because every case below is rejected."""

    def __init__(self, numel, dtype, device="cuda:0", contiguous=True, cuda=True):
        import torch
        self._n, self.dtype, self.device = numel, dtype, torch.device(device)
        self._c, self.is_cuda = contiguous, cuda

    def numel(self):
        return self._n

    def is_contiguous(self):
        return self._c

    def data_ptr(self):
        return BASE


def _binding_case(**over):
    torch = pytest.importorskip("torch")
    L = capi.fsdp_layout(capi.FSDP_PER_PARAM, 2, [(64, 8)], capi.FSDP_BF16, capi.FSDP_BF16)
    P, S = L.full_numel, L.shard_numel
    args = dict(shard=[FakeTensor(S, torch.bfloat16) for _ in range(2)],
                full_out=[FakeTensor(P, torch.bfloat16) for _ in range(2)])
    args.update({k: v(torch, P, S) for k, v in over.items()})
    return L, args


@pytest.mark.parametrize("over,needle", [
    (dict(full_out=lambda t, P, S: [FakeTensor(P - 1, t.bfloat16), FakeTensor(P, t.bfloat16)]),
     "elements"),
    (dict(shard=lambda t, P, S: [FakeTensor(S, t.bfloat16), FakeTensor(S - 8, t.bfloat16)]),
     "elements"),
    (dict(full_out=lambda t, P, S: [FakeTensor(P, t.float32), FakeTensor(P, t.bfloat16)]),
     "dtype"),
    (dict(shard=lambda t, P, S: [FakeTensor(S, t.bfloat16, "cuda:1"),
                                 FakeTensor(S, t.bfloat16)]), "is on"),
    (dict(shard=lambda t, P, S: [FakeTensor(S, t.bfloat16, contiguous=False),
                                 FakeTensor(S, t.bfloat16)]), "contiguous"),
    (dict(shard=lambda t, P, S: [FakeTensor(S, t.bfloat16)]), "expected 2"),
    (dict(shard=lambda t, P, S: [FakeTensor(S, t.bfloat16, "cpu", cuda=False),
                                 FakeTensor(S, t.bfloat16)]), "not a CUDA tensor"),
])
def test_binding_checks_tensor_size_dtype_device(lib, over, needle):
    L, a = _binding_case(**over)
    with pytest.raises(capi.FsdpArgumentError) as e:
        capi.fsdp_all_gather_unflatten(L, a["shard"], a["full_out"])
    assert e.value.status == capi.FSDP_EINVAL and needle in str(e.value)


def test_binding_checks_reduce_scatter_state_dtypes(lib):
    torch = pytest.importorskip("torch")
    L = capi.fsdp_layout(capi.FSDP_PER_PARAM, 2, [(64, 8)], capi.FSDP_BF16, capi.FSDP_BF16)
    P, S = L.full_numel, L.shard_numel
    f32 = lambda n: [FakeTensor(n, torch.float32) for _ in range(2)]
    b16 = lambda n: [FakeTensor(n, torch.bfloat16) for _ in range(2)]
    hp = _hp()
    # fp32 gradients for a bf16-gradient layout
    with pytest.raises(capi.FsdpArgumentError, match="grad_full"):
        capi.fsdp_reduce_scatter_adamw(L, f32(P), f32(S), f32(S), f32(S), b16(S), None, hp, 1)
    # bf16 master
    with pytest.raises(capi.FsdpArgumentError, match="master"):
        capi.fsdp_reduce_scatter_adamw(L, b16(P), b16(S), f32(S), f32(S), b16(S), None, hp, 1)
    # a short second moment
    with pytest.raises(capi.FsdpArgumentError, match=r"v\[1\]"):
        capi.fsdp_reduce_scatter_adamw(L, b16(P), f32(S), f32(S), [f32(S)[0], f32(S - 1)[0]],
                                       b16(S), None, hp, 1)
    # accumulators must be fp32 and full-unit sized
    with pytest.raises(capi.FsdpArgumentError, match="acc_full"):
        capi.fsdp_reduce_scatter_adamw_accum(L, f32(P - 8), b16(P), f32(S), f32(S), f32(S),
                                             b16(S), None, hp, 1)
    with pytest.raises(capi.FsdpArgumentError, match="out"):
        capi.fsdp_all_reduce(L, b16(P), b16(P - 1), capi.FSDP_BF16)


def test_unit_step_advances_only_on_accepted_calls(lib):
    torch = pytest.importorskip("torch")
    from fully_sharded_state_gb300 import unit as unit_mod

    class Stub(unit_mod.ShardedUnit):
        def __init__(self):  # no device buffers: only the step bookkeeping is exercised
            self.layout = capi.fsdp_layout(capi.FSDP_PER_PARAM, 2, [(64, 8)], capi.FSDP_BF16,
                                           capi.FSDP_BF16)
            S = self.layout.shard_numel
            self.master = self.m = self.v = [FakeTensor(S, torch.float32) for _ in range(2)]
            self.param_shard = [FakeTensor(S, torch.bfloat16) for _ in range(2)]
            self.step = 4

    U = Stub()
    short = [FakeTensor(1, torch.bfloat16) for _ in range(2)]
    with pytest.raises(capi.FsdpArgumentError):
        U.reduce_scatter_adamw(short, _hp())
    assert U.step == 4
    with pytest.raises(capi.FsdpArgumentError):
        U.reduce_scatter_adamw_accum(short, short, _hp())
    assert U.step == 4


# ---- several units per call --------------------------------------------------

def _units_rs(lib, layouts, R, over=None, bytes_per=1 << 22):
    n = len(layouts)
    k = iter(range(10_000))
    arr = lambda: _ptrs([BASE + next(k) * bytes_per for _ in range(n * R)])
    a = dict(grad=arr(), master=arr(), m=arr(), v=arr(), pshard=arr(), gshard=None, hp=_hp(),
             step=1)
    a.update(over or {})
    lay = _ptrs([L.handle for L in layouts])
    return lib.fsdp_reduce_scatter_adamw_units(n, lay, a["grad"], a["master"], a["m"], a["v"],
                                               a["pshard"], a["gshard"], ctypes.byref(a["hp"]),
                                               a["step"], None)


def test_units_calls_reject_bad_arguments(lib):
    A = capi.fsdp_layout(capi.FSDP_FLAT, 4, [(512, 512)], capi.FSDP_BF16, capi.FSDP_BF16)
    B8 = capi.fsdp_layout(capi.FSDP_FLAT, 8, [(512, 512)], capi.FSDP_BF16, capi.FSDP_BF16)
    F = capi.fsdp_layout(capi.FSDP_FLAT, 4, [(512, 512)], capi.FSDP_F32, capi.FSDP_BF16)
    MB = 1 << 22
    sh = _ptrs([BASE + k * MB for k in range(8)])
    fo = _ptrs([BASE + (100 + k) * MB for k in range(8)])
    g = lambda *Ls: _ptrs([L.handle for L in Ls])
    assert lib.fsdp_all_gather_unflatten_units(0, g(A), sh, fo, None) == capi.FSDP_EINVAL
    assert lib.fsdp_all_gather_unflatten_units(2, None, sh, fo, None) == capi.FSDP_EINVAL
    assert lib.fsdp_all_gather_unflatten_units(2, _ptrs([A.handle, 0]), sh, fo,
                                               None) == capi.FSDP_EINVAL
    # mixed R or dtypes
    assert lib.fsdp_all_gather_unflatten_units(2, g(A, B8), sh, fo, None) == capi.FSDP_EINVAL
    assert lib.fsdp_all_gather_unflatten_units(2, g(A, F), sh, fo, None) == capi.FSDP_EINVAL
    # unit 1's destination 2 (entry 6) overlaps unit 0's destination 0
    bad = _ptrs([BASE + (100 + k) * MB for k in range(6)] + [BASE + 100 * MB + 64,
                                                            BASE + 200 * MB])
    assert lib.fsdp_all_gather_unflatten_units(2, g(A, A), sh, bad, None) == capi.FSDP_EINVAL
    assert b"full_out" in lib.fsdp_last_error()
    # a misaligned pointer is reported by its index in the whole array
    bad = _ptrs([BASE + (100 + k) * MB for k in range(5)] + [BASE + 300 * MB + 2,
                                                            BASE + 301 * MB, BASE + 302 * MB])
    assert lib.fsdp_all_gather_unflatten_units(2, g(A, A), sh, bad, None) == capi.FSDP_EALIGN
    assert b"full_out[5]" in lib.fsdp_last_error()
    # the reduce-scatter: bf16 layouts need param_shard_out; F32 layouts take none
    assert _units_rs(lib, [A, A], 4, dict(pshard=None)) == capi.FSDP_EINVAL
    assert _units_rs(lib, [F, F], 4) == capi.FSDP_EINVAL
    assert _units_rs(lib, [A, A], 4, dict(step=0)) == capi.FSDP_EINVAL
    assert _units_rs(lib, [A, B8], 4) == capi.FSDP_EINVAL


def test_units_calls_skip_empty_units(lib):
    E = capi.fsdp_layout(capi.FSDP_PER_PARAM, 4, [(0, 8)], capi.FSDP_BF16, capi.FSDP_BF16)
    nul = _ptrs([0] * 8)
    lay = _ptrs([E.handle, E.handle])
    assert lib.fsdp_all_gather_unflatten_units(2, lay, nul, nul, None) == capi.FSDP_OK
    assert lib.fsdp_reduce_scatter_adamw_units(2, lay, nul, nul, nul, nul, nul, None,
                                               ctypes.byref(_hp()), 1, None) == capi.FSDP_OK


def test_write_stream_rejects_bad_arguments(lib):
    MB = 1 << 20
    d = _ptrs([BASE, BASE + MB])
    assert lib.fsdp_write_stream(None, 2, 1024, 0, None) == capi.FSDP_EINVAL
    assert lib.fsdp_write_stream(d, 0, 1024, 0, None) == capi.FSDP_EINVAL
    assert lib.fsdp_write_stream(d, 2, 1000, 0, None) == capi.FSDP_EINVAL  # not 32-byte chunks
    assert lib.fsdp_write_stream(_ptrs([BASE + 16, BASE + MB]), 2, 1024, 0,
                                 None) == capi.FSDP_EALIGN
    # overlapping destinations
    assert lib.fsdp_write_stream(_ptrs([BASE, BASE + 512]), 2, 1024, 0, None) == capi.FSDP_EINVAL
    assert lib.fsdp_write_stream(d, 2, 0, 0, None) == capi.FSDP_OK
