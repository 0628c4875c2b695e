"""The equivalence recipe of "FSDP2 的参数全聚合、梯度归约分片与显存峰值", §12,
over several training steps of a small model.

Path A: one device, fp32, the whole batch, torch.optim.AdamW.
Path B: R virtual ranks. Every step gathers the unit with the library's
all-gather, each rank runs forward and backward (torch autograd; the model's
compute is not part of the shard engine) on its equal slice of the batch with
the gathered parameters, and the library's reduce-scatter + AdamW turns the R
local gradients into the sharded update. With equal slices the average of the
ranks' mean losses is the whole batch's mean loss (§04's assumption), so both
paths take the same steps; after each one the gathered parameters must match
path A to torch.testing.assert_close(rtol=1e-5, atol=1e-7).
"""
import pytest
import torch

from fully_sharded_state_gb300 import AdamWHP, ShardedUnit

pytestmark = pytest.mark.gpu

SHAPES = [(64, 32), (64,), (16, 64), (16,)]   # W1, b1, W2, b2
LR, WD = 1e-3, 0.01


def forward(params, x):
    w1, b1, w2, b2 = params
    return torch.tanh(x @ w1.t() + b1) @ w2.t() + b2


@pytest.mark.parametrize("mode,R", [("per_param", 2), ("flat", 4), ("zero3", 4),
                                    ("per_param", 8)])
def test_sharded_training_matches_single_device(cuda_lib, mode, R, monkeypatch):
    # both paths in full fp32 matmuls (no TF32)
    monkeypatch.setattr(torch.backends.cuda.matmul, "allow_tf32", False)
    torch.manual_seed(0)
    dev = torch.device("cuda")
    init = [torch.randn(s, device=dev) * 0.1 for s in SHAPES]
    batch = 8 * R
    xs = [torch.randn(batch, 32, device=dev) for _ in range(5)]
    ys = [torch.randn(batch, 16, device=dev) for _ in range(5)]

    # path A
    ref = [torch.nn.Parameter(t.clone()) for t in init]
    opt = torch.optim.AdamW(ref, lr=LR, betas=(0.9, 0.999), eps=1e-8, weight_decay=WD)

    # path B
    U = ShardedUnit(SHAPES, R, mode, "f32", "f32", names=["w1", "b1", "w2", "b2"])
    U.shard_from_full(torch.cat([t.reshape(-1) for t in init]))
    full = U.alloc_full()
    hp = AdamWHP(LR, 0.9, 0.999, 1e-8, WD)

    for step, (x, y) in enumerate(zip(xs, ys)):
        opt.zero_grad()
        torch.nn.functional.mse_loss(forward(ref, x), y).backward()
        opt.step()

        U.all_gather(full)
        grads = []
        for r in range(R):
            views = U.unflatten(full[r])
            local = [views[k].detach().clone().requires_grad_(True)
                     for k in ("w1", "b1", "w2", "b2")]
            sl = slice(r * 8, (r + 1) * 8)
            torch.nn.functional.mse_loss(forward(local, x[sl]), y[sl]).backward()
            grads.append(torch.cat([p.grad.reshape(-1) for p in local]))
        U.reduce_scatter_adamw(grads, hp)

        U.all_gather(full)
        got = U.unflatten(full[0])
        for k, p in zip(("w1", "b1", "w2", "b2"), ref):
            torch.testing.assert_close(got[k], p.detach(), rtol=1e-5, atol=1e-7,
                                       msg=lambda m: f"step {step} {k}: {m}")
