"""Two more GPU checks.

Guards: every output buffer sits inside a larger allocation whose bytes
before and after it hold a known pattern; after pack, gather, reduce-scatter
+ AdamW (with and without accumulators, register and staged kernels),
all-reduce, ZeRO-1's AdamW from the averaged gradient and accumulation the
patterns must be intact, so no kernel writes
outside its buffers.

Equivalence ("FSDP2 的参数全聚合、梯度归约分片与显存峰值", §12): one sharded
step equals one step of torch.optim.AdamW on the full parameters with the
rank-averaged gradient, to torch.testing.assert_close(rtol=1e-5, atol=1e-7).
"""
import numpy as np
import pytest
import torch

from fully_sharded_state_gb300 import AdamWHP, ShardedUnit, capi

pytestmark = pytest.mark.gpu
GUARD = 4096  # bytes each side


class Guarded:
    """Tensors of `numel` elements placed GUARD bytes into a patterned block."""

    def __init__(self):
        self.blocks = []

    def __call__(self, numel, dtype):
        es = torch.tensor([], dtype=dtype).element_size()
        blk = torch.empty(2 * GUARD + numel * es + 16, dtype=torch.uint8, device="cuda")
        blk.fill_(0xA5)
        self.blocks.append((blk, numel * es))
        return blk[GUARD:GUARD + numel * es].view(dtype)

    def check(self):
        torch.cuda.synchronize()
        for blk, nb in self.blocks:
            assert torch.all(blk[:GUARD] == 0xA5)
            assert torch.all(blk[GUARD + nb:] == 0xA5)


@pytest.mark.parametrize("mode,pdt,gdt,R,shapes", [
    ("per_param", "bf16", "bf16", 4, [(1001, 3), (7, 513), (0, 5), (1, 64)]),
    ("flat", "bf16", "f32", 3, [(1001, 3), (5, 7)]),
    ("zero3", "f32", "bf16", 8, [(127, 513), (3, 1), (4097, 1), (9,)]),
    ("per_param", "f32", "f32", 9, [(2049, 1), (33, 8)]),
    # 24.6M parameters: large enough for the reduce-scatter that stages its
    # gradient slices in shared memory; rows of 4,097 put most rank pieces
    # off the 8-element grid, so staged and register tiles share the launch
    ("per_param", "bf16", "bf16", 8, [(6000, 4097), (7, 513), (64,)]),
    ("per_param", "bf16", "f32", 4, [(6000, 4097), (5, 3)]),
])
def test_kernels_write_only_inside_their_buffers(cuda_lib, mode, pdt, gdt, R, shapes):
    G = Guarded()
    U = ShardedUnit(shapes, R, mode, pdt, gdt)
    P, S = U.P, U.S
    tp = torch.bfloat16 if pdt == "bf16" else torch.float32
    tg = torch.bfloat16 if gdt == "bf16" else torch.float32
    U.master = [G(S, torch.float32) for _ in range(R)]
    U.m = [G(S, torch.float32).zero_() for _ in range(R)]
    U.v = [G(S, torch.float32).zero_() for _ in range(R)]
    U.param_shard = [G(S, torch.bfloat16) for _ in range(R)] if pdt == "bf16" else None
    U.shard_from_full(torch.randn(P, device="cuda"))
    grads = [G(P, tg).copy_(torch.randn(P, device="cuda")) for _ in range(R)]
    full = [G(P, tp) for _ in range(R)]
    U.all_gather(full)
    hp = AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01)
    gsh = [G(S, torch.float32) for _ in range(R)]
    U.reduce_scatter_adamw(grads, hp, grad_shard_out=gsh)
    acc = [G(P, torch.float32) for _ in range(R)]
    U.accumulate_grad(grads, acc, first=True)
    U.accumulate_grad(grads, acc, first=False)
    U.reduce_scatter_adamw_accum(acc, grads, hp)
    ar = [G(P, torch.float32) for _ in range(R)]
    U.all_reduce(grads, ar, "f32")
    U.adamw_from_reduced(ar, hp)
    ar16 = [G(P, torch.bfloat16) for _ in range(R)]
    U.all_reduce(grads, ar16, "bf16")
    G.check()


@pytest.mark.parametrize("R,gdt", [(2, "f32"), (4, "bf16"), (8, "bf16")])
def test_one_sharded_step_equals_single_device_adamw(cuda_lib, R, gdt):
    shapes = [(512,), (512, 512), (2048, 512)]
    U = ShardedUnit(shapes, R, "per_param", "f32", gdt)
    w = torch.randn(U.P, device="cuda") * 0.02
    U.shard_from_full(w)
    tg = torch.bfloat16 if gdt == "bf16" else torch.float32
    grads = [(torch.randn(U.P, device="cuda") * 1e-3).to(tg) for _ in range(R)]
    lr, wd = 1e-3, 0.01
    U.reduce_scatter_adamw(grads, AdamWHP(lr, 0.9, 0.999, 1e-8, wd))
    full = U.alloc_full()
    U.all_gather(full)

    p = torch.nn.Parameter(w.clone())
    p.grad = torch.stack([g.float() for g in grads]).mean(0)
    opt = torch.optim.AdamW([p], lr=lr, betas=(0.9, 0.999), eps=1e-8, weight_decay=wd)
    opt.step()
    torch.testing.assert_close(full[0], p.detach(), rtol=1e-5, atol=1e-7)
