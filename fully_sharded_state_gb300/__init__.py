"""GB300-native FSDP per-unit shard engine.

dim-0 sharding (FSDP1 FlatParameter or FSDP2 per-parameter), parameter
all-gather + unflatten, and the fixed-order fp32 gradient reduce-scatter
fused with the sharded AdamW step, over R virtual ranks held in one GPU's
HBM. The compute path is the CUDA library ``_lib/libfsdp_shard.so``
(C ABI in ``include/fsdp_shard.h``); ``capi`` binds it with ctypes.
"""
from .capi import (FSDP_BF16, FSDP_F32, FSDP_FLAT, FSDP_PER_PARAM, FSDP_ZERO3, AdamWHP, FsdpError,
                   LibraryNotBuilt, fsdp_accumulate_grad, fsdp_all_gather_unflatten,
                   fsdp_all_reduce, fsdp_reduce_scatter_adamw_accum, fsdp_layout, fsdp_pack_flat,
                   fsdp_reduce_scatter_adamw, fsdp_reduce_scatter_adamw_gather, fsdp_version)

__all__ = ["FSDP_BF16", "FSDP_F32", "FSDP_FLAT", "FSDP_PER_PARAM", "FSDP_ZERO3", "AdamWHP", "FsdpError",
           "LibraryNotBuilt", "fsdp_accumulate_grad", "fsdp_all_gather_unflatten",
           "fsdp_all_reduce", "fsdp_reduce_scatter_adamw_accum", "fsdp_layout", "fsdp_pack_flat",
           "fsdp_reduce_scatter_adamw", "fsdp_reduce_scatter_adamw_gather", "fsdp_version",
           "ShardedUnit"]


def __getattr__(name):
    if name == "ShardedUnit":  # imports torch; keep the package importable without it
        from .unit import ShardedUnit
        return ShardedUnit
    raise AttributeError(name)
