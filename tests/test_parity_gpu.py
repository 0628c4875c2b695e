"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Every workload that the oracle finishes in seconds is run whole: the pages'
toy, the 512/8/2048 block (FSDP2), twelve blocks as FSDP1 FlatParameters and
the ragged stress unit; then edge cases: R = 1, odd R, the generic-R kernels,
empty parameters and ranks, misaligned rank boundaries, more parameters than
one launch takes, mixed dtypes, P = 0."""
import pytest
import torch

from fully_sharded_state_gb300 import synth
from parity import UnitCase, run_accumulation_case, run_overlap_case, run_unit_case

pytestmark = pytest.mark.gpu


def _workload_case(name, u, step=1, prior=False):
    wl = synth.WORKLOADS[name]
    case = UnitCase(shapes=wl.unit_shapes(u), R=wl.R, mode=wl.mode, param_dtype=wl.param_dtype,
                    grad_dtype=wl.grad_dtype, seed=wl.cfg, w_std=wl.w_std, g_std=wl.g_std,
                    step=step, hp=(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay))
    w = synth.host_weights(wl, u)
    grads = synth.host_grads(wl, u)
    moments = None
    if prior:
        from fully_sharded_state_gb300 import ShardedUnit
        S = ShardedUnit(case.shapes, case.R, case.mode, case.param_dtype, case.grad_dtype).S
        moments = synth.host_moments(wl, u, S)
    return case, w, grads, moments


@pytest.mark.parametrize("u", [0, 1])
def test_toy_walkthrough_units(cuda_lib, u):
    case, w, g, _ = _workload_case("toy", u)
    run_unit_case(case, w, g)


@pytest.mark.parametrize("step,prior", [(1, False), (3, True)])
def test_block_512_fsdp2(cuda_lib, step, prior):
    case, w, g, mom = _workload_case("block", 0, step, prior)
    res = run_unit_case(case, w, g, mom)
    assert res["P"] == 3_146_752


def test_twelve_blocks_fsdp1_flat(cuda_lib):
    for u in range(12):
        case, w, g, mom = _workload_case("block12_flat", u, step=2, prior=True)
        run_unit_case(case, w, g, mom)


@pytest.mark.parametrize("step,prior", [(1, False), (2, True)])
def test_ragged_stress(cuda_lib, step, prior):
    case, w, g, mom = _workload_case("ragged", 0, step, prior)
    run_unit_case(case, w, g, mom)


EDGE = {
    "R1": UnitCase([(37, 5), (8,)], R=1),
    "R3_odd_average": UnitCase([(1000, 24), (7, 3)], R=3, seed=3),
    "R5_generic": UnitCase([(513, 64), (1,)], R=5, seed=5),
    "R9_generic_flat": UnitCase([(300, 70), (11, 13)], R=9, mode="flat", seed=9),
    "R16_generic": UnitCase([(4097, 8)], R=16, seed=16, step=4, prior_moments=True),
    "R64_max": UnitCase([(200, 16), (3,)], R=64, seed=64),
    "empty_params_and_ranks": UnitCase([(0, 8), (1, 513), (3, 1), (5, 64), (0, 0), (2, 2)], R=8,
                                       seed=11),
    "odd_width_bf16": UnitCase([(129, 513), (127, 1)], R=4, seed=12),
    "flat_ragged_tail": UnitCase([(1001, 3), (5, 7)], R=4, mode="flat", seed=13),
    "flat_smaller_than_R": UnitCase([(3,)], R=8, mode="flat", seed=14),
    "tile_edges": UnitCase([(2048, 1), (2049, 1), (2047, 1), (1, 2048 * 3 + 8)], R=2, seed=15),
    "many_params_several_launches": UnitCase([((k * 7) % 13 + 1, 8 + (k % 3)) for k in range(600)],
                                             R=8, seed=17),
    "f32_params_bf16_grads": UnitCase([(256, 40), (9,)], R=4, param_dtype="f32", seed=18),
    "bf16_params_f32_grads": UnitCase([(256, 40), (9,)], R=4, grad_dtype="f32", seed=19,
                                      outlier_frac=0.01),
    "f32_flat_outliers": UnitCase([(4097, 3)], R=8, mode="flat", param_dtype="f32",
                                  grad_dtype="f32", g_std=1.0, w_std=1.0, outlier_frac=0.01,
                                  seed=20),
    "tiny_gradients_eps_dominated": UnitCase([(64, 64)], R=4, g_std=1e-9, seed=21),
    "no_weight_decay_large_lr": UnitCase([(64, 64)], R=2, hp=(0.1, 0.8, 0.99, 1e-6, 0.0),
                                         step=5, prior_moments=True, seed=22),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(cuda_lib, name):
    run_unit_case(EDGE[name])


def test_empty_unit_is_a_no_op(cuda_lib):
    from fully_sharded_state_gb300 import AdamWHP, ShardedUnit
    U = ShardedUnit([(0, 4), (0,)], R=4)
    assert U.P == 0
    U.all_gather(U.alloc_full())
    U.reduce_scatter_adamw(U.alloc_grads(), AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01))
    torch.cuda.synchronize()


def test_side_stream(cuda_lib):
    """Calls are asynchronous on the caller's stream."""
    from fully_sharded_state_gb300 import ShardedUnit
    U = ShardedUnit([(4096, 256)], R=4)
    w = torch.randn(U.P, device="cuda")
    s = torch.cuda.Stream()
    full = U.alloc_full()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        U.shard_from_full(w, stream=s)
        U.all_gather(full, stream=s)
    s.synchronize()
    want = w.to(torch.bfloat16)
    for d in range(4):
        assert torch.equal(full[d].view(torch.int16), want.view(torch.int16))


def test_device_errors_launch_nothing(cuda_lib):
    import ctypes
    from fully_sharded_state_gb300 import FsdpError, ShardedUnit, capi
    U = ShardedUnit([(64, 64)], R=2)
    full = U.alloc_full()
    # a bf16 view one element in: not 16-byte aligned
    big = torch.empty(U.P + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(FsdpError) as e:
        capi.fsdp_all_gather_unflatten(U.layout, U.gather_sources(), [big[1:U.P + 1], full[1]])
    assert e.value.status == capi.FSDP_EALIGN
    # two destinations that are the same buffer
    with pytest.raises(FsdpError) as e:
        capi.fsdp_all_gather_unflatten(U.layout, U.gather_sources(), [full[0], full[0]])
    assert e.value.status == capi.FSDP_EINVAL
    # output in pinned host memory is rejected before any launch
    pinned = [torch.empty(U.P, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    lib = capi.load()
    arr_in = (ctypes.c_void_p * 2)(*[t.data_ptr() for t in U.gather_sources()])
    arr_out = (ctypes.c_void_p * 2)(*[t.data_ptr() for t in pinned])
    st = lib.fsdp_all_gather_unflatten(U.layout.handle, arr_in, arr_out, None)
    assert st == capi.FSDP_EINVAL
    torch.cuda.synchronize()


def test_native_library_is_loaded(cuda_lib):
    maps = open("/proc/self/maps").read()
    assert "libfsdp_shard.so" in maps


OVERLAP = {
    "block_and_block": (EDGE["odd_width_bf16"], UnitCase([(512,), (512, 512), (2048, 512)], R=4)),
    "ragged_fp32_pair": (UnitCase([(1001, 3), (7, 513), (1, 64)], R=8, param_dtype="f32",
                                  grad_dtype="f32", g_std=1.0, w_std=1.0, outlier_frac=0.01),
                         UnitCase([(127, 513), (3, 1), (4097, 1)], R=8, param_dtype="f32",
                                  grad_dtype="f32")),
    "flat_rs_per_param_gather": (UnitCase([(1001, 3), (5, 7)], R=4, mode="flat"),
                                 UnitCase([(300, 70)], R=4)),
    "generic_R5": (UnitCase([(513, 64), (9,)], R=5), UnitCase([(77, 40)], R=5)),
    "tiny_rs_big_gather": (UnitCase([(3,)], R=2), UnitCase([(4096, 64)], R=2)),
    "different_R": (UnitCase([(256, 40)], R=4), UnitCase([(256, 40)], R=8)),
    "different_dtype": (UnitCase([(256, 40)], R=4), UnitCase([(256, 40)], R=4,
                                                            param_dtype="f32")),
    "many_params": (EDGE["many_params_several_launches"], UnitCase([(64, 8)], R=8)),
}


@pytest.mark.parametrize("name", sorted(OVERLAP))
def test_prefetch_reduce_scatter_then_gather(cuda_lib, name):
    run_overlap_case(*OVERLAP[name])


def test_prefetch_rejects_gathering_the_updated_unit(cuda_lib):
    from fully_sharded_state_gb300 import AdamWHP, FsdpError, ShardedUnit
    U = ShardedUnit([(64, 64)], R=2)
    with pytest.raises(FsdpError):
        U.reduce_scatter_adamw_and_gather(U.alloc_grads(), AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01),
                                          U, U.alloc_full())


ALL_REDUCE = {
    "block_bf16_to_f32": (UnitCase([(512,), (512, 512), (2048, 512)], R=4), "f32"),
    "bf16_to_bf16_R8": (UnitCase([(4097, 8), (3,)], R=8, seed=31), "bf16"),
    "f32_R3_outliers": (UnitCase([(1001, 5)], R=3, grad_dtype="f32", param_dtype="f32",
                                 g_std=1.0, outlier_frac=0.01, seed=32), "f32"),
    "R1_copy": (UnitCase([(77, 13)], R=1, seed=33), "f32"),
    "ragged_tail_generic_R6": (UnitCase([(2049, 3), (5,)], R=6, seed=34), "bf16"),
}


@pytest.mark.parametrize("name", sorted(ALL_REDUCE))
def test_all_reduce(cuda_lib, name):
    import oracle
    from fully_sharded_state_gb300 import ShardedUnit
    from parity import assert_bits_equal, host, host_inputs, to_dev
    case, out_dt = ALL_REDUCE[name]
    _, grads = host_inputs(case)
    U = ShardedUnit(case.shapes, case.R, case.mode, case.param_dtype, case.grad_dtype)
    tdt = torch.bfloat16 if out_dt == "bf16" else torch.float32
    out = [torch.zeros(U.P, dtype=tdt, device="cuda") for _ in range(case.R)]
    U.all_reduce([to_dev(g) for g in grads], out, out_dt)
    want = oracle.all_reduce(grads, out_bf16=out_dt == "bf16")
    for d in range(case.R):
        assert_bits_equal(host(out[d]), want[d], f"all-reduce out[{d}]")


@pytest.mark.parametrize("mode", ["per_param", "flat"])
def test_all_reduce_equals_gather_of_reduce_scatter(cuda_lib, mode):
    """On the GPU: gathering the fp32 reduce-scatter shards gives the
    all-reduce output bit for bit."""
    from fully_sharded_state_gb300 import AdamWHP, ShardedUnit
    from parity import host_inputs, to_dev
    case = UnitCase([(1001, 3), (257, 64), (9,)], R=4, mode=mode, seed=35)
    _, grads = host_inputs(case)
    g = [to_dev(x) for x in grads]
    U = ShardedUnit(case.shapes, 4, mode, "bf16", "bf16")
    gsh = [torch.zeros(U.S, dtype=torch.float32, device="cuda") for _ in range(4)]
    U.reduce_scatter_adamw(g, AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01), grad_shard_out=gsh)
    F = ShardedUnit(case.shapes, 4, mode, "f32", "bf16")   # same layout, fp32 shards
    gathered = F.alloc_full()
    from fully_sharded_state_gb300 import capi
    capi.fsdp_all_gather_unflatten(F.layout, gsh, gathered)
    out = [torch.empty(U.P, dtype=torch.float32, device="cuda") for _ in range(4)]
    U.all_reduce(g, out, "f32")
    for d in range(4):
        assert torch.equal(gathered[d].view(torch.int32), out[d].view(torch.int32))


ACCUM = {
    "block_K3": (UnitCase([(512,), (512, 512), (2048, 512)], R=4, seed=41), 3),
    "ragged_fp32_K2": (UnitCase([(1001, 3), (7, 513), (1, 64)], R=8, param_dtype="f32",
                                grad_dtype="f32", g_std=1.0, w_std=1.0, outlier_frac=0.01,
                                seed=42), 2),
    "flat_K4": (UnitCase([(1001, 3), (5, 7)], R=4, mode="flat", seed=43), 4),
    "generic_R5_K2": (UnitCase([(513, 64), (9,)], R=5, seed=44, step=3), 2),
    "single_micro_batch": (UnitCase([(300, 70)], R=2, seed=45), 1),
}


@pytest.mark.parametrize("name", sorted(ACCUM))
def test_gradient_accumulation(cuda_lib, name):
    run_accumulation_case(*ACCUM[name])


ZERO3 = {
    "block_R4": UnitCase([(512,), (512, 512), (512, 512), (512, 512), (512, 512), (512,),
                          (512, 2048), (2048, 512)], R=4, mode="zero3", seed=51),
    "ragged_fp32_R8": UnitCase([(1001, 3), (7, 513), (1, 64), (4097, 1), (127, 513), (3, 1)], R=8,
                               mode="zero3", param_dtype="f32", grad_dtype="f32", g_std=1.0,
                               w_std=1.0, outlier_frac=0.01, seed=52),
    "more_ranks_than_tensors": UnitCase([(300, 70), (9,)], R=6, mode="zero3", seed=53),
    "R1": UnitCase([(37, 5), (8,)], R=1, mode="zero3", seed=54),
    "many_params_step3": UnitCase([((k * 7) % 13 + 1, 8 + (k % 3)) for k in range(300)], R=8,
                                  mode="zero3", seed=55, step=3, prior_moments=True),
}


@pytest.mark.parametrize("name", sorted(ZERO3))
def test_zero3_inter_tensor(cuda_lib, name):
    run_unit_case(ZERO3[name])


def test_zero3_prefetch_and_accumulation(cuda_lib):
    run_overlap_case(ZERO3["block_R4"], UnitCase([(256, 40), (33, 8)], R=4, mode="zero3"))
    run_accumulation_case(UnitCase([(513, 64), (9,), (77, 40)], R=4, mode="zero3", seed=56), 3)
