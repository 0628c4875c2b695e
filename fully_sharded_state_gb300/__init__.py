"""GB300-native FSDP per-unit shard engine.

dim-0 sharding (FSDP1 FlatParameter or FSDP2 per-parameter), parameter
all-gather + unflatten, and the fixed-order fp32 gradient reduce-scatter
fused with the sharded AdamW step, over R virtual ranks held in one GPU's
HBM. The compute path is the CUDA library ``_lib/libfsdp_shard.so``
(C ABI in ``include/fsdp_shard.h``); ``capi`` binds it with ctypes.
"""
from .capi import (FSDP_BF16, FSDP_F32, FSDP_FLAT, FSDP_PER_PARAM, FSDP_ZERO3, AdamWHP, FsdpError,
                   FsdpArgumentError, LibraryNotBuilt, fsdp_accumulate_grad,
                   fsdp_adamw_from_reduced,
                   fsdp_all_gather_unflatten, fsdp_all_gather_unflatten_units, fsdp_all_reduce,
                   fsdp_reduce_scatter_adamw_accum, fsdp_layout, fsdp_pack_flat,
                   fsdp_reduce_scatter_adamw, fsdp_reduce_scatter_adamw_gather,
                   fsdp_reduce_scatter_adamw_units, fsdp_stage_wait_selftest, fsdp_stage_wait_timeouts,
                   fsdp_version, PreparedCall,
                   prepare_fsdp_all_gather_unflatten, prepare_fsdp_all_gather_unflatten_units,
                   prepare_fsdp_reduce_scatter_adamw, prepare_fsdp_reduce_scatter_adamw_units)

__all__ = ["FSDP_BF16", "FSDP_F32", "FSDP_FLAT", "FSDP_PER_PARAM", "FSDP_ZERO3", "AdamWHP", "FsdpError",
           "FsdpArgumentError", "LibraryNotBuilt", "fsdp_accumulate_grad", "fsdp_adamw_from_reduced",
           "fsdp_all_gather_unflatten", "fsdp_all_gather_unflatten_units", "fsdp_all_reduce",
           "fsdp_reduce_scatter_adamw_accum", "fsdp_layout", "fsdp_pack_flat",
           "fsdp_reduce_scatter_adamw", "fsdp_reduce_scatter_adamw_gather",
           "fsdp_reduce_scatter_adamw_units", "fsdp_stage_wait_selftest", "fsdp_stage_wait_timeouts", "fsdp_version",
           "PreparedCall",
           "prepare_fsdp_all_gather_unflatten", "prepare_fsdp_all_gather_unflatten_units",
           "prepare_fsdp_reduce_scatter_adamw", "prepare_fsdp_reduce_scatter_adamw_units",
           "ShardedUnit",
           "all_gather_units", "reduce_scatter_adamw_units", "prepare_all_gather_units",
           "prepare_reduce_scatter_adamw_units"]


def __getattr__(name):
    # these import torch; keep the package importable without it
    if name in ("ShardedUnit", "all_gather_units", "reduce_scatter_adamw_units",
                "prepare_all_gather_units", "prepare_reduce_scatter_adamw_units"):
        from . import unit
        return getattr(unit, name)
    raise AttributeError(name)
