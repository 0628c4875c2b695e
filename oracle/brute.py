"""Pure-Python brute force of the shard engine for tiny integer-valued cases.

TEST INFRASTRUCTURE (part of the oracle). Written from the pages' own
formulation, with Python lists and slicing, independently of the C oracle,
so that each can catch a mistake in the other:

- shard: ``t[start:end]`` with ``s = ceil(d0 / R)``, ``start = r*s``,
  ``end = min(start + s, d0)`` ("从源码理解 FSDP", §2.1 partition);
- gather: concatenate the non-empty shards in rank order ("从源码理解 FSDP",
  §2.2 gather_tensor);
- FlatParameter: concat(flatten(p_i)), padded to a multiple of R, cut into R
  equal pieces ("FSDP Transformer Block Sharding Example", FSDP1);
- reduce-scatter: element-wise sum over ranks, rank r keeps segment r
  ("FSDP2 的参数全聚合、梯度归约分片与显存峰值", §09).

Values are Python ints or exact rationals; nothing here rounds.
"""
from __future__ import annotations


def shard_dim0(rows: list, R: int, r: int) -> list:
    """Rank r's dim-0 slice of a tensor given as a list of rows."""
    d0 = len(rows)
    s = -(-d0 // R)
    start = r * s
    end = min(start + s, d0)
    return rows[start:end]


def gather_dim0(shards: list) -> list:
    """Full tensor (list of rows) from all ranks' slices, in rank order."""
    full = []
    for sh in shards:
        if len(sh) > 0:
            full.extend(sh)
    return full


def as_rows(flat: list, shape: tuple) -> list:
    """View a flat list as dim-0 rows of a tensor of `shape`."""
    d0 = shape[0] if len(shape) else 1
    inner = 1
    for x in shape[1:]:
        inner *= x
    return [flat[k * inner:(k + 1) * inner] for k in range(d0)]


def per_param_shards(params: list, shapes: list, R: int) -> list:
    """FSDP2: for each rank, the list of its slices (each a list of rows)."""
    return [[shard_dim0(as_rows(p, shp), R, r) for p, shp in zip(params, shapes)]
            for r in range(R)]


def flat_shards(params: list, R: int) -> list:
    """FSDP1: the R equal pieces of the zero-padded FlatParameter."""
    flat = [x for p in params for x in p]
    S = -(-len(flat) // R)
    flat = flat + [0] * (R * S - len(flat))
    return [flat[r * S:(r + 1) * S] for r in range(R)]


def flat_gather(pieces: list, numel: int) -> list:
    flat = [x for piece in pieces for x in piece]
    return flat[:numel]


def reduce_scatter_sum(grads: list, R: int, owner_ranges: list) -> list:
    """grads[q] = rank q's full flat gradient; owner_ranges[r] = the flat
    index ranges rank r keeps. Returns, per rank, the summed values."""
    total = [sum(grads[q][j] for q in range(R)) for j in range(len(grads[0]))]
    return [[total[j] for (a, b) in owner_ranges[r] for j in range(a, b)] for r in range(R)]


def per_param_owner_ranges(shapes: list, R: int) -> list:
    """Flat index ranges [a, b) of the full unit that each rank owns (FSDP2)."""
    out = [[] for _ in range(R)]
    base = 0
    for shp in shapes:
        d0 = shp[0] if len(shp) else 1
        inner = 1
        for x in shp[1:]:
            inner *= x
        rows = list(range(d0))
        for r in range(R):
            mine = shard_dim0(rows, R, r)
            if mine and inner > 0:
                out[r].append((base + mine[0] * inner, base + (mine[-1] + 1) * inner))
        base += d0 * inner
    return out


def zero3_parts(numels: list, R: int) -> list:
    """ZeRO-3 inter-tensor partition ("从源码理解 FSDP", §2.1): whole tensors,
    in order, go to the current part, which is closed once it holds at least
    ceil(total/R) elements (the last part takes the rest). Returns the
    list of tensor indices of every part."""
    target = -(-sum(numels) // R)
    parts = [[] for _ in range(R)]
    cur, filled = 0, 0
    for i, n in enumerate(numels):
        parts[cur].append(i)
        filled += n
        if filled >= target and cur < R - 1:
            cur, filled = cur + 1, 0
    return parts
