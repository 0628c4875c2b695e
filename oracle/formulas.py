"""The pages' memory and communication formulas, written out.

TEST INFRASTRUCTURE (part of the oracle). Each function states one formula
and cites where it comes from; the tests pin them to the numbers the pages
print.
"""
from __future__ import annotations

from fractions import Fraction


# --- communication -------------------------------------------------------

def ring_volume_per_rank(numel: int, R: int) -> Fraction:
    """Elements one rank sends in an all-gather or a reduce-scatter of a
    `numel`-element tensor over R ranks: (R-1)/R * numel.
    ("FSDP Transformer Block Sharding Example", All-Gather mechanism: per-GPU
    send = (N-1)/N x layer size.)"""
    return Fraction(R - 1, R) * numel


def allreduce_volume_per_rank(numel: int, R: int) -> Fraction:
    """DDP all-reduce: 2(R-1)/R * numel per rank ("FSDP Training Step
    Walkthrough", per-step communication summary, the DDP comparison)."""
    return 2 * Fraction(R - 1, R) * numel


def fsdp_step_tally(layer_numels: list, R: int) -> list:
    """One FSDP training step's collectives, in schedule order, as
    (phase, op, layer, elements sent per rank).

    Schedule ("FSDP Training Step Walkthrough", Steps 1-6): forward gathers
    each layer in order; backward walks the layers in reverse, re-gathering
    each layer and then reduce-scattering its gradient; the optimizer step
    communicates nothing."""
    tally = []
    for k, n in enumerate(layer_numels):
        tally.append(("forward", "all-gather", k, ring_volume_per_rank(n, R)))
    for k in reversed(range(len(layer_numels))):
        n = layer_numels[k]
        tally.append(("backward", "all-gather", k, ring_volume_per_rank(n, R)))
        tally.append(("backward", "reduce-scatter", k, ring_volume_per_rank(n, R)))
    tally.append(("optimizer", "none", -1, Fraction(0)))
    return tally


# --- memory ----------------------------------------------------------------

def ddp_state_bytes(P, b_w, b_g, b_o):
    """M_DDP = P (b_w + b_g + b_o) ("FSDP2 的参数全聚合、梯度归约分片与显存峰值", §01)."""
    return P * (b_w + b_g + b_o)


def shard_state_bytes(P, b_w, b_g, b_o, R):
    """M_shard ~= P (b_w + b_g + b_o) / R (same page, §01)."""
    return Fraction(ddp_state_bytes(P, b_w, b_g, b_o)) / R


def peak_bytes(m_shard, largest_unsharded, prefetch, activations=0, temp=0):
    """M_peak ~= M_shard + M_largest_unsharded + M_prefetch + M_a + M_temp
    (same page, §01)."""
    return m_shard + largest_unsharded + prefetch + activations + temp


def ddp_bytes_per_param_adamw_mixed():
    """Per-parameter bytes of DDP with fp16 params + fp32 master and AdamW
    ("从源码理解 FSDP", §1.1): params (fp16 + fp32 master) 6, grads 2 (fp16),
    AdamW m and v 8 (fp32) -> 16."""
    params = 2 + 4
    grads = 2
    optim = 4 + 4
    return params + grads + optim


def zero3_bytes_per_param(R):
    """ZeRO-3 / FSDP: every item sharded, 16P/N ("从源码理解 FSDP", §1.2, §3.2)."""
    return Fraction(ddp_bytes_per_param_adamw_mixed(), R)


# --- the 512/8/2048 TransformerBlock ----------------------------------------

def block_shapes(hidden=512, ffn=2048, with_norms=True):
    """Parameter shapes of one block in the page's tree order
    ("FSDP Transformer Block Sharding Example", model definition):
    norm1, W_Q, W_K, W_V, W_O, norm2, W_up, W_down. W_up is taken as
    [hidden, ffn] exactly as the page's table prints it."""
    shapes = []
    if with_norms:
        shapes.append(("norm1", (hidden,)))
    shapes += [("W_Q", (hidden, hidden)), ("W_K", (hidden, hidden)),
               ("W_V", (hidden, hidden)), ("W_O", (hidden, hidden))]
    if with_norms:
        shapes.append(("norm2", (hidden,)))
    shapes += [("W_up", (hidden, ffn)), ("W_down", (ffn, hidden))]
    return shapes


def numel(shape):
    n = 1
    for x in shape:
        n *= x
    return n
