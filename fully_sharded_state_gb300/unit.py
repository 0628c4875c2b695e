"""One FSDP unit sharded over R virtual ranks held in this GPU's HBM.

The user-facing wrapper over the C ABI, in the spirit of wrapping one
Transformer block as an FSDP unit ("FSDP Transformer Block Sharding
Example", wrapping granularity): torch allocates the per-rank buffers; every
data movement and every update runs in the CUDA library.

Per rank r the unit keeps: ``master[r]`` (fp32 master shard), ``m[r]`` and
``v[r]`` (AdamW moments, fp32, zero at start), and for bf16 parameters
``param_shard[r]`` (the bf16 shard the all-gather reads).
"""
from __future__ import annotations

import torch

from . import capi

_DT = {"bf16": (capi.FSDP_BF16, torch.bfloat16), "f32": (capi.FSDP_F32, torch.float32)}
_MODE = {"flat": capi.FSDP_FLAT, "per_param": capi.FSDP_PER_PARAM, "zero3": capi.FSDP_ZERO3}


class ShardedUnit:
    def __init__(self, shapes, R: int, mode: str = "per_param", param_dtype: str = "bf16",
                 grad_dtype: str = "bf16", device="cuda", names=None):
        self.shapes = [tuple(int(x) for x in s) for s in shapes]
        self.names = list(names) if names is not None else [f"p{i}" for i in range(len(shapes))]
        self.R = R
        self.mode = mode
        self.param_dtype, self.grad_dtype = param_dtype, grad_dtype
        self.device = torch.device(device)
        self.layout = capi.fsdp_layout(_MODE[mode], R, self.shapes, _DT[param_dtype][0],
                                       _DT[grad_dtype][0])
        self.P = self.layout.full_numel
        self.S = self.layout.shard_numel
        z = lambda dt: [torch.zeros(self.S, dtype=dt, device=self.device) for _ in range(R)]
        self.master = z(torch.float32)
        self.m = z(torch.float32)
        self.v = z(torch.float32)
        self.param_shard = z(torch.bfloat16) if param_dtype == "bf16" else None
        self.step = 0

    # -- buffers ------------------------------------------------------------
    @property
    def param_torch_dtype(self):
        return _DT[self.param_dtype][1]

    @property
    def grad_torch_dtype(self):
        return _DT[self.grad_dtype][1]

    def gather_sources(self):
        """The shard buffers the all-gather reads (bf16 shard, or the fp32 master)."""
        return self.param_shard if self.param_shard is not None else self.master

    def alloc_full(self):
        """R full-unit buffers in the parameter dtype (one per destination rank)."""
        return [torch.empty(self.P, dtype=self.param_torch_dtype, device=self.device)
                for _ in range(self.R)]

    def alloc_grads(self):
        return [torch.empty(self.P, dtype=self.grad_torch_dtype, device=self.device)
                for _ in range(self.R)]

    def unflatten(self, full) -> dict:
        """Views of one full-unit buffer as the original parameters (no copy)."""
        out = {}
        for i, (name, shape) in enumerate(zip(self.names, self.shapes)):
            off = self.layout.param_full_offset(i)
            n = 1
            for x in shape:
                n *= x
            out[name] = full[off:off + n].view(shape)
        return out

    # -- the hot path ---------------------------------------------------------
    def shard_from_full(self, full_f32, stream=None) -> None:
        capi.fsdp_pack_flat(self.layout, full_f32, self.param_shard, self.master, stream)

    def all_gather(self, full_out, stream=None) -> None:
        capi.fsdp_all_gather_unflatten(self.layout, self.gather_sources(), full_out, stream)

    def _next_step(self, step):
        return self.step + 1 if step is None else int(step)

    def reduce_scatter_adamw(self, grads, hp: capi.AdamWHP, grad_shard_out=None,
                             step: int | None = None, stream=None) -> None:
        """One optimizer step from the R ranks' full local gradients. The
        step count advances only when the call is accepted."""
        t = self._next_step(step)
        capi.fsdp_reduce_scatter_adamw(self.layout, grads, self.master, self.m, self.v,
                                       self.param_shard, grad_shard_out, hp, t, stream)
        self.step = t

    def reduce_scatter_adamw_and_gather(self, grads, hp: capi.AdamWHP, other: "ShardedUnit",
                                        other_full, grad_shard_out=None, step: int | None = None,
                                        stream=None) -> None:
        """This unit's optimizer step, then the all-gather of `other` (a different
        unit, e.g. the next one to be computed), validated together."""
        t = self._next_step(step)
        capi.fsdp_reduce_scatter_adamw_gather(
            self.layout, grads, self.master, self.m, self.v, self.param_shard, grad_shard_out,
            hp, t, other.layout, other.gather_sources(), other_full, stream)
        self.step = t

    def all_reduce(self, grads, out, out_dtype: str = "f32", stream=None) -> None:
        """DDP's all-reduce of the R full gradients into R full outputs
        (fp32 or bf16), for comparison with the sharded path."""
        capi.fsdp_all_reduce(self.layout, grads, out, _DT[out_dtype][0], stream)

    def adamw_from_reduced(self, grad_avg_full, hp: capi.AdamWHP, step: int | None = None,
                           stream=None) -> None:
        """ZeRO-1's optimizer step: every rank updates its own elements from
        its full averaged fp32 gradient (all_reduce's fp32 output). The step
        count advances as with reduce_scatter_adamw."""
        t = self._next_step(step)
        capi.fsdp_adamw_from_reduced(self.layout, grad_avg_full, self.master, self.m, self.v,
                                     self.param_shard, hp, t, stream)
        self.step = t

    # -- prepared calls (checked once, re-issued every step) -----------------
    def prepare_all_gather(self, full_out):
        """The all-gather into ``full_out`` with its arguments bound; call the
        result (optionally with ``stream=``) to issue it."""
        return capi.prepare_fsdp_all_gather_unflatten(self.layout, self.gather_sources(),
                                                      full_out)

    def prepare_reduce_scatter_adamw(self, grads, grad_shard_out=None):
        """The reduce-scatter + AdamW step on ``grads`` with its arguments
        bound. Call the result with ``hp`` (and ``step=``, ``stream=``); the
        step count advances as with reduce_scatter_adamw."""
        call = capi.prepare_fsdp_reduce_scatter_adamw(self.layout, grads, self.master, self.m,
                                                      self.v, self.param_shard, grad_shard_out)

        def run(hp: capi.AdamWHP, step: int | None = None, stream=None) -> None:
            t = self._next_step(step)
            call(hp, t, stream)
            self.step = t
        return run

    # -- gradient accumulation over micro-batches ---------------------------
    def alloc_accumulators(self):
        """R fp32 full-unit gradient accumulators."""
        return [torch.empty(self.P, dtype=torch.float32, device=self.device)
                for _ in range(self.R)]

    def accumulate_grad(self, grads, acc, first: bool, stream=None) -> None:
        """acc = grads (first micro-batch) or acc + grads, per rank, in fp32."""
        capi.fsdp_accumulate_grad(self.layout, acc, grads, first, stream)

    def reduce_scatter_adamw_accum(self, acc, grads, hp: capi.AdamWHP, grad_shard_out=None,
                                   step: int | None = None, stream=None) -> None:
        """The optimizer step on acc + grads (the last micro-batch fused in)."""
        t = self._next_step(step)
        capi.fsdp_reduce_scatter_adamw_accum(self.layout, acc, grads, self.master, self.m,
                                             self.v, self.param_shard, grad_shard_out, hp, t,
                                             stream)
        self.step = t


# -- several units per launch --------------------------------------------------

def all_gather_units(units, full_outs, stream=None) -> None:
    """The all-gather + unflatten of every unit in ``units`` (same R and
    dtypes) in one launch; ``full_outs[u]`` is unit u's list of R outputs."""
    capi.fsdp_all_gather_unflatten_units([U.layout for U in units],
                                         [U.gather_sources() for U in units], full_outs, stream)


def reduce_scatter_adamw_units(units, grads, hp: capi.AdamWHP, grad_shard_outs=None,
                               step: int | None = None, stream=None) -> None:
    """One optimizer step of every unit in ``units`` in one launch. All units
    take the same step count: one past the first unit's, or ``step``."""
    t = units[0]._next_step(step)
    bf16 = units[0].param_shard is not None
    capi.fsdp_reduce_scatter_adamw_units(
        [U.layout for U in units], grads, [U.master for U in units], [U.m for U in units],
        [U.v for U in units], [U.param_shard for U in units] if bf16 else None,
        grad_shard_outs, hp, t, stream)
    for U in units:
        U.step = t



def prepare_all_gather_units(units, full_outs):
    """all_gather_units with its arguments bound once (see PreparedCall)."""
    return capi.prepare_fsdp_all_gather_unflatten_units([U.layout for U in units],
                                                        [U.gather_sources() for U in units],
                                                        full_outs)


def prepare_reduce_scatter_adamw_units(units, grads, grad_shard_outs=None):
    """reduce_scatter_adamw_units with its arguments bound once; call the
    result with ``hp`` (and ``step=``, ``stream=``)."""
    bf16 = units[0].param_shard is not None
    call = capi.prepare_fsdp_reduce_scatter_adamw_units(
        [U.layout for U in units], grads, [U.master for U in units], [U.m for U in units],
        [U.v for U in units], [U.param_shard for U in units] if bf16 else None, grad_shard_outs)

    def run(hp: capi.AdamWHP, step: int | None = None, stream=None) -> None:
        t = units[0]._next_step(step)
        call(hp, t, stream)
        for U in units:
            U.step = t
    return run
