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
