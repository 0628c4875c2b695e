"""Seeded synthetic inputs shaped like the FSDP pages' workloads.

This module only draws random numbers and names shapes. It holds no part of
the shard engine's arithmetic (no layout, gather, reduction or optimizer
math), so that both the CUDA path and the CPU oracle can be fed from it.

Workloads (all FSDP units, R virtual ranks):

- ``toy``: two layers, each one fp32 vector of length 4, R=2
  ("FSDP Training Step Walkthrough", Setup).
- ``block``: one TransformerBlock hidden=512, heads=8, ffn=2048 with its two
  LayerNorm scales, FSDP2 per-parameter, R=4, bf16 params and grads
  ("FSDP Transformer Block Sharding Example", model definition).
- ``block12_flat``: twelve such blocks, one FSDP1 FlatParameter unit each, R=4.
- ``ragged``: 64 fp32 tensors with dim 0 from {1,3,5,7,127,1000,1001,4097}
  and dim 1 from {1,64,513}, R=8; 1 % of gradient entries scaled by 1e4.
- ``llama4``: four Llama-style decoder blocks (hidden 4096, ffn 14336, GQA
  with 1024-wide K/V), one FSDP unit per block, R=8, bf16 params and grads.

Seeds: weights 1000+cfg, gradients 2000+cfg+101*rank, outlier masks
3000+cfg+101*rank, prior first moments 4000+cfg, prior second moments
5000+cfg; each plus 7919*unit.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

try:  # torch is only needed for bf16 conversion and device-side generation
    import torch
except ImportError:  # pragma: no cover
    torch = None


@dataclass(frozen=True)
class Workload:
    name: str
    cfg: int
    mode: str                 # "flat" (FSDP1) or "per_param" (FSDP2)
    R: int
    units: tuple              # per unit: tuple of (param name, shape)
    param_dtype: str          # "bf16" or "f32"
    grad_dtype: str           # "bf16" or "f32"
    w_std: float
    g_std: float
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    lr: float = 1e-3
    betas: tuple = (0.9, 0.999)
    eps: float = 1e-8
    weight_decay: float = 0.01
    notes: str = field(default="", compare=False)

    def unit_shapes(self, u: int) -> list:
        return [shape for _, shape in self.units[u]]

    def unit_numel(self, u: int) -> int:
        return int(sum(int(np.prod(s, dtype=np.int64)) for s in self.unit_shapes(u)))


def _block_512():
    h, f = 512, 2048
    return (("norm1", (h,)), ("W_Q", (h, h)), ("W_K", (h, h)), ("W_V", (h, h)),
            ("W_O", (h, h)), ("norm2", (h,)), ("W_up", (h, f)), ("W_down", (f, h)))


def _llama_block():
    h, f, kv = 4096, 14336, 1024
    return (("W_q", (h, h)), ("W_k", (kv, h)), ("W_v", (kv, h)), ("W_o", (h, h)),
            ("W_gate", (f, h)), ("W_up", (f, h)), ("W_down", (h, f)),
            ("attn_norm", (h,)), ("ffn_norm", (h,)))


def _ragged_shapes(cfg=4, n=64):
    rng = np.random.default_rng(1000 + cfg)
    d0 = rng.choice(np.array([1, 3, 5, 7, 127, 1000, 1001, 4097]), size=n)
    d1 = rng.choice(np.array([1, 64, 513]), size=n)
    return tuple((f"t{k}", (int(a), int(b))) for k, (a, b) in enumerate(zip(d0, d1)))


WORKLOADS = {
    "toy": Workload("toy", 1, "per_param", 2, ((("W1", (4,)),), (("W2", (4,)),)),
                    "f32", "f32", 1.0, 1.0),
    "block": Workload("block", 2, "per_param", 4, (_block_512(),), "bf16", "bf16", 0.02, 1e-3),
    "block12_flat": Workload("block12_flat", 3, "flat", 4, tuple(_block_512() for _ in range(12)),
                             "bf16", "bf16", 0.02, 1e-3),
    "ragged": Workload("ragged", 4, "per_param", 8, (_ragged_shapes(),), "f32", "f32", 1.0, 1.0,
                       outlier_frac=0.01, outlier_scale=1e4),
    "llama4": Workload("llama4", 5, "per_param", 8, tuple(_llama_block() for _ in range(4)),
                       "bf16", "bf16", 0.02, 1e-3),
}


def seed(role: str, wl: Workload, unit: int = 0, rank: int = 0) -> int:
    base = {"w": 1000, "g": 2000, "mask": 3000, "m": 4000, "v": 5000}[role]
    extra = 101 * rank if role in ("g", "mask") else 0
    return base + wl.cfg + extra + 7919 * unit


# ---- host (numpy) ----------------------------------------------------------

def host_normal(s: int, n: int, std: float) -> np.ndarray:
    x = np.random.default_rng(s).standard_normal(n, dtype=np.float32)
    return (x * np.float32(std)).astype(np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 with torch (a library conversion) and
    return the bit patterns as uint16."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def host_weights(wl: Workload, u: int) -> np.ndarray:
    """Full fp32 weights of unit u, parameters concatenated in unit order."""
    return host_normal(seed("w", wl, u), wl.unit_numel(u), wl.w_std)


def host_grads(wl: Workload, u: int) -> list:
    """Each rank's full local gradient of unit u (uint16 bf16 bits or float32)."""
    out = []
    n = wl.unit_numel(u)
    for r in range(wl.R):
        g = host_normal(seed("g", wl, u, r), n, wl.g_std)
        if wl.outlier_frac > 0:
            mask = np.random.default_rng(seed("mask", wl, u, r)).random(n) < wl.outlier_frac
            g[mask] *= np.float32(wl.outlier_scale)
        out.append(to_bf16_bits(g) if wl.grad_dtype == "bf16" else g)
    return out


def host_moments(wl: Workload, u: int, n: int):
    """Plausible AdamW moments from earlier steps, n per rank buffer:
    m ~ N(0, (0.1 g_std)^2), v = 1e-3 * (g_std z)^2 (non-negative)."""
    ms, vs = [], []
    for r in range(wl.R):
        ms.append(host_normal(seed("m", wl, u) + 13 * r, n, 0.1 * wl.g_std))
        z = host_normal(seed("v", wl, u) + 13 * r, n, wl.g_std)
        vs.append((np.float32(1e-3) * z * z).astype(np.float32))
    return ms, vs


# ---- device (torch) ----------------------------------------------------------

def _dev_gen(s: int, device):
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def device_normal(s: int, n: int, std: float, device, dtype=None):
    x = torch.randn(n, generator=_dev_gen(s, device), device=device, dtype=torch.float32)
    x.mul_(std)
    return x if dtype is None else x.to(dtype)


def device_weights(wl: Workload, u: int, device):
    return device_normal(seed("w", wl, u), wl.unit_numel(u), wl.w_std, device)


def device_grads(wl: Workload, u: int, device) -> list:
    dt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    out = []
    n = wl.unit_numel(u)
    for r in range(wl.R):
        g = device_normal(seed("g", wl, u, r), n, wl.g_std, device)
        if wl.outlier_frac > 0:
            mask = torch.rand(n, generator=_dev_gen(seed("mask", wl, u, r), device),
                              device=device) < wl.outlier_frac
            g[mask] *= wl.outlier_scale
        out.append(g.to(dt))
    return out


def device_moments(wl: Workload, u: int, n: int, device):
    ms, vs = [], []
    for r in range(wl.R):
        ms.append(device_normal(seed("m", wl, u) + 13 * r, n, 0.1 * wl.g_std, device))
        z = device_normal(seed("v", wl, u) + 13 * r, n, wl.g_std, device)
        vs.append(z.mul_(z).mul_(1e-3))
    return ms, vs
