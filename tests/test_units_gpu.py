"""Several FSDP units per call (fsdp_all_gather_unflatten_units,
fsdp_reduce_scatter_adamw_units) against the oracle, unit by unit, and the
binding's refusal of a tensor too short for the layout, with guard bytes
around it showing that nothing was written."""
import pytest
import torch

from fully_sharded_state_gb300 import AdamWHP, FsdpArgumentError, ShardedUnit, synth
from parity import UnitCase, run_units_case

pytestmark = pytest.mark.gpu


def _block12():
    wl = synth.WORKLOADS["block12_flat"]
    return [UnitCase(wl.unit_shapes(u), wl.R, "flat", seed=40 + u) for u in range(12)]


CASES = {
    # the twelve 512/8/2048 blocks as FSDP1 units, R = 4: one launch (48 pointers)
    "block12_flat": (_block12(), 1),
    # twenty such units: 80 pointers per array, so two launches
    "block20_flat_two_launches": ([UnitCase([(512,), (512, 512), (2048, 512)], 4, "flat",
                                            seed=90 + u) for u in range(20)], 2),
    # FSDP2 units, ragged fp32 with outliers, R = 8, an empty unit among them
    "ragged_f32_R8": ([UnitCase([(1001, 3), (7, 513), (1, 64)], 8, param_dtype="f32",
                                grad_dtype="f32", w_std=1.0, g_std=1.0, outlier_frac=0.01,
                                seed=7),
                       UnitCase([(0, 5)], 8, param_dtype="f32", grad_dtype="f32"),
                       UnitCase([(127, 513), (3, 1), (4097, 1)], 8, param_dtype="f32",
                                grad_dtype="f32", seed=8)], 3),
    # more than 256 parameters over the units: the segments span launches
    "many_params": ([UnitCase([(17, 9)] * 150, 2, seed=60 + u) for u in range(3)], 1),
    # ZeRO-3 owners and a generic R
    "zero3_R5": ([UnitCase([(300, 70), (9,), (40, 40)], 5, "zero3", seed=70 + u)
                  for u in range(4)], 1),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_units_match_oracle(cuda_lib, name):
    cases, step = CASES[name]
    run_units_case(cases, step=step)


def test_units_share_one_layout(cuda_lib):
    cases = [UnitCase([(512, 64), (64,)], 4, seed=80 + u) for u in range(6)]
    run_units_case(cases, share_layout=True)


def test_units_equal_one_unit_calls(cuda_lib):
    """The multi-unit step gives the same bits as one call per unit."""
    from fully_sharded_state_gb300 import all_gather_units, reduce_scatter_adamw_units
    wl = synth.WORKLOADS["block12_flat"]
    dev = torch.device("cuda")
    hp = AdamWHP(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay)
    sets = []
    for _ in range(2):
        units, grads = [], []
        for u in range(len(wl.units)):
            U = ShardedUnit(wl.unit_shapes(u), wl.R, "flat")
            U.shard_from_full(synth.device_normal(synth.seed("w", wl, u), U.P, wl.w_std, dev))
            units.append(U)
            grads.append([synth.device_normal(synth.seed("g", wl, u, r), U.P, wl.g_std, dev,
                                              torch.bfloat16) for r in range(wl.R)])
        sets.append((units, grads))
    (A, gA), (B, gB) = sets
    fullA = [U.alloc_full() for U in A]
    fullB = [U.alloc_full() for U in B]
    for _ in range(3):
        all_gather_units(A, fullA)
        reduce_scatter_adamw_units(A, gA, hp)
        for k, U in enumerate(B):
            U.all_gather(fullB[k])
            U.reduce_scatter_adamw(gB[k], hp)
    torch.cuda.synchronize()
    for UA, UB, fa, fb in zip(A, B, fullA, fullB):
        assert UA.step == UB.step == 3
        for r in range(wl.R):
            for x, y in ((UA.master[r], UB.master[r]), (UA.m[r], UB.m[r]), (UA.v[r], UB.v[r])):
                assert torch.equal(x.view(torch.int32), y.view(torch.int32))
            assert torch.equal(UA.param_shard[r].view(torch.int16),
                               UB.param_shard[r].view(torch.int16))
            assert torch.equal(fa[r].view(torch.int16), fb[r].view(torch.int16))


def test_short_view_is_refused_before_any_write(cuda_lib):
    """A destination one element short of the unit, placed at the start of a
    guarded allocation: the binding refuses it and no byte changes."""
    U = ShardedUnit([(1024, 64)], R=2)
    guard = 4096
    blk = torch.full((2 * guard + U.P * 2,), 0xA5, dtype=torch.uint8, device="cuda")
    short = blk[guard:guard + (U.P - 1) * 2].view(torch.bfloat16)
    full = U.alloc_full()
    with pytest.raises(FsdpArgumentError) as e:
        U.all_gather([short, full[1]])
    assert "elements" in str(e.value)
    g32 = [torch.zeros(U.P, device="cuda") for _ in range(2)]  # fp32 for a bf16-grad layout
    with pytest.raises(FsdpArgumentError):
        U.reduce_scatter_adamw(g32, AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01))
    assert U.step == 0
    torch.cuda.synchronize()
    assert torch.all(blk == 0xA5)


def test_host_memory_inputs_are_refused(cuda_lib):
    """Every buffer must be device memory: pinned host memory passed as a
    shard (an input) is refused by the C library before any launch."""
    import ctypes
    from fully_sharded_state_gb300 import capi
    U = ShardedUnit([(64, 64)], R=2)
    full = U.alloc_full()
    pinned = [torch.empty(U.S, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    lib = capi.load()
    arr_in = (ctypes.c_void_p * 2)(*[t.data_ptr() for t in pinned])
    arr_out = (ctypes.c_void_p * 2)(*[t.data_ptr() for t in full])
    st = lib.fsdp_all_gather_unflatten(U.layout.handle, arr_in, arr_out, None)
    assert st == capi.FSDP_EINVAL
    assert b"not device memory" in lib.fsdp_last_error()
    torch.cuda.synchronize()


@pytest.mark.parametrize("pdt", ["bf16", "f32"])
def test_sixteen_byte_aligned_buffers(cuda_lib, pdt):
    """Buffers that are 16-byte but not 32-byte aligned (views 16 bytes into
    an allocation) take the kernels' 16-byte-vector paths; the results are
    the oracle's, bit for bit, and equal those of aligned buffers."""
    import numpy as np

    import oracle
    from parity import host, to_dev
    R = 4
    shapes = [(512, 64), (96, 40), (7, 513)]
    U = ShardedUnit(shapes, R, "per_param", pdt, "bf16")
    O = oracle.layout(oracle.PER_PARAM, R, shapes)
    w = synth.host_normal(5, U.P, 0.02)
    U.shard_from_full(to_dev(w))
    masters, p16 = oracle.pack(O, w, with_bf16=pdt == "bf16")
    tp = torch.bfloat16 if pdt == "bf16" else torch.float32

    def offset_views(n, dtype, count):
        bufs = [torch.zeros(n + 64, dtype=dtype, device="cuda") for _ in range(count)]
        return bufs, [b[16 // torch.tensor([], dtype=dtype).element_size():][:n] for b in bufs]

    # shards moved into 16-byte offset views, destinations likewise
    _, sh = offset_views(U.S, tp, R)
    for r in range(R):
        sh[r].copy_(U.gather_sources()[r])
    _, full = offset_views(U.P, tp, R)
    assert all(t.data_ptr() % 32 == 16 for t in sh + full)
    from fully_sharded_state_gb300 import capi
    capi.fsdp_all_gather_unflatten(U.layout, sh, full)
    want = oracle.all_gather(O, p16 if pdt == "bf16" else masters)
    for d in range(R):
        np.testing.assert_array_equal(host(full[d]).view(np.uint8), want[d].view(np.uint8))
    # all-reduce into 16-byte offset fp32 outputs equals the aligned result
    g = [to_dev(x) for x in synth.host_grads(synth.WORKLOADS["block"], 0)[:R]]
    gP = [x[:U.P].contiguous() for x in g]
    _, out_off = offset_views(U.P, torch.float32, R)
    out_al = [torch.empty(U.P, dtype=torch.float32, device="cuda") for _ in range(R)]
    U.all_reduce(gP, out_off, "f32")
    U.all_reduce(gP, out_al, "f32")
    want = oracle.all_reduce([host(x) for x in gP], out_bf16=False)
    for d in range(R):
        assert torch.equal(out_off[d].view(torch.int32), out_al[d].view(torch.int32))
        np.testing.assert_array_equal(host(out_al[d]).view(np.uint32), want[d].view(np.uint32))
    torch.cuda.synchronize()


def test_write_stream_helper_writes_exactly_its_buffers(cuda_lib):
    """The write-stream measurement helper fills each buffer with its
    pattern and nothing around it."""
    from fully_sharded_state_gb300 import capi
    n, nbytes, guard = 3, 1 << 20, 4096
    blk = [torch.full((nbytes + 2 * guard,), 0xA5, dtype=torch.uint8, device="cuda")
           for _ in range(n)]
    dst = [b[guard:guard + nbytes].view(torch.float32) for b in blk]
    capi.fsdp_write_stream(dst, pattern=0x3F800000)
    torch.cuda.synchronize()
    for b, d in zip(blk, dst):
        assert torch.all(d == 1.0)
        assert torch.all(b[:guard] == 0xA5) and torch.all(b[guard + nbytes:] == 0xA5)


def test_prepared_calls_equal_plain_calls(cuda_lib):
    """A prepared call (arguments checked and marshalled once) gives the same
    bits as the plain call, step after step, and keeps its tensors alive."""
    import gc
    shapes = [(300, 64), (17, 9), (64,)]
    hp = AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01)
    A = ShardedUnit(shapes, 4)
    B = ShardedUnit(shapes, 4)
    w = torch.randn(A.P, device="cuda") * 0.02
    A.shard_from_full(w)
    B.shard_from_full(w)
    grads = [(torch.randn(A.P, device="cuda") * 1e-3).to(torch.bfloat16) for _ in range(4)]
    fa, fb = A.alloc_full(), B.alloc_full()
    gather = A.prepare_all_gather(fa)
    step = A.prepare_reduce_scatter_adamw([g.clone() for g in grads])
    del fa
    gc.collect()
    for _ in range(3):
        gather()
        step(hp)
        B.all_gather(fb)
        B.reduce_scatter_adamw(grads, hp)
    gather()
    B.all_gather(fb)
    torch.cuda.synchronize()
    assert A.step == B.step == 3
    held = gather._tensors[2]  # the prepared call's own reference to its outputs
    for r in range(4):
        assert torch.equal(A.master[r].view(torch.int32), B.master[r].view(torch.int32))
        assert torch.equal(held[r].view(torch.int16), fb[r].view(torch.int16))
