"""ZeRO-1's step against the FSDP step ("从源码理解 FSDP", §1.2, the ZeRO
stages): all-reduce the R gradients (every rank gets the averaged fp32
gradient), let each rank update its own partition from its own copy
(fsdp_adamw_from_reduced), then all-gather. The all-reduce folds the ranks in
the reduce-scatter's order and the update is the same code, so every buffer
must equal the fused reduce-scatter + AdamW step's bit for bit; that path is
compared with the oracle element by element elsewhere."""
import pytest
import torch

from fully_sharded_state_gb300 import AdamWHP, ShardedUnit, synth

pytestmark = pytest.mark.gpu

CASES = [
    ("per_param", "bf16", "bf16", 4, [(1001, 3), (7, 513), (0, 5), (1, 64), (2049, 64)]),
    ("flat", "bf16", "f32", 3, [(1001, 3), (5, 7)]),
    ("zero3", "f32", "bf16", 8, [(127, 513), (3, 1), (4097, 1), (9,)]),
    ("per_param", "f32", "f32", 8, [(4096, 513), (1000, 1001)]),
    # 21M parameters: the fused path takes the staged kernel here
    ("per_param", "bf16", "bf16", 8, [(4096, 4096), (1024, 4096), (4096,)]),
]


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("mode,pdt,gdt,R,shapes", CASES)
def test_zero1_step_equals_the_fsdp_step(cuda_lib, mode, pdt, gdt, R, shapes):
    dev = torch.device("cuda")
    units = [ShardedUnit(shapes, R, mode, pdt, gdt) for _ in range(2)]
    P, S = units[0].P, units[0].S
    w = synth.device_normal(31, P, 0.02, dev)
    for U in units:
        U.shard_from_full(w)
        for r in range(R):  # moments of a previous step
            U.m[r].copy_(synth.device_normal(40 + r, S, 1e-4, dev))
            U.v[r].copy_(synth.device_normal(50 + r, S, 1e-3, dev).square_().mul_(1e-3))
    tg = torch.bfloat16 if gdt == "bf16" else torch.float32
    grads = [synth.device_normal(60 + r, P, 1e-3, dev, tg) for r in range(R)]
    hp = AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01)

    z1, fsdp = units
    avg = [torch.empty(P, dtype=torch.float32, device=dev) for _ in range(R)]
    z1.all_reduce(grads, avg, "f32")
    z1.adamw_from_reduced(avg, hp, step=3)
    fsdp.reduce_scatter_adamw(grads, hp, step=3)
    assert z1.step == fsdp.step == 3
    for r in range(R):
        for a, b, what in ((z1.master[r], fsdp.master[r], "master"), (z1.m[r], fsdp.m[r], "m"),
                           (z1.v[r], fsdp.v[r], "v")):
            assert torch.equal(_bits(a), _bits(b)), f"{what}[{r}]"
        if pdt == "bf16":
            assert torch.equal(_bits(z1.param_shard[r]), _bits(fsdp.param_shard[r])), r
    # the all-gather that follows shares the updated partitions
    f1, f2 = z1.alloc_full(), fsdp.alloc_full()
    z1.all_gather(f1)
    fsdp.all_gather(f2)
    for d in range(R):
        assert torch.equal(_bits(f1[d]), _bits(f2[d])), d
