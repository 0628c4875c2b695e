"""Helpers of the GPU parity tests: run one FSDP unit through the CUDA path
(via the C ABI) and through the CPU oracle on the same seeded inputs, and
compare element by element.

The bars:
  - pack, all-gather and the fp32 reduce-scatter shard: bit-exact;
  - AdamW master: |d| <= 1e-5 * max(1, |w|) per step;
  - AdamW moments: |d| <= 1e-5 * |want| + 1e-30 (relative);
  - bf16 parameter shard: within 1 bf16 ulp.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import oracle
from fully_sharded_state_gb300 import AdamWHP, ShardedUnit
from fully_sharded_state_gb300 import synth

MASTER_RTOL = 1e-5
MOMENT_RTOL = 1e-5
BF16_ULP = 1


def to_dev_bf16(bits: np.ndarray, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def to_dev(x: np.ndarray, device="cuda"):
    if x.dtype == np.uint16:
        return to_dev_bf16(x, device)
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def host(t) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between bit patterns (sign-magnitude ordered)."""
    def key(u):
        x = u.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(key(a) - key(b))


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str):
    g = got.view(np.uint16 if got.dtype in (np.uint16, np.int16) else np.uint32)
    w = want.view(np.uint16 if want.dtype in (np.uint16, np.int16) else np.uint32)
    bad = np.flatnonzero(g != w)
    assert bad.size == 0, f"{what}: {bad.size} of {g.size} differ, first at {bad[:5]}"


def assert_master_close(got, want, what="master"):
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    bound = MASTER_RTOL * np.maximum(1.0, np.abs(want.astype(np.float64)))
    bad = np.flatnonzero(~(err <= bound))
    assert bad.size == 0, f"{what}: {bad.size} beyond 1e-5*max(1,|w|), first {bad[:5]}"


def assert_moment_close(got, want, what):
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    bound = MOMENT_RTOL * np.abs(want.astype(np.float64)) + 1e-30
    bad = np.flatnonzero(~(err <= bound))
    assert bad.size == 0, f"{what}: {bad.size} beyond the relative bound, first {bad[:5]}"


def assert_bf16_close(got, want, what="bf16 shard"):
    d = bf16_ulp_diff(got, want)
    assert d.max(initial=0) <= BF16_ULP, f"{what}: max {d.max()} ulp"


def omode(mode: str) -> int:
    return {"flat": oracle.FLAT, "per_param": oracle.PER_PARAM, "zero3": oracle.ZERO3}[mode]


@dataclass
class UnitCase:
    shapes: list
    R: int
    mode: str = "per_param"      # or "flat", "zero3"
    param_dtype: str = "bf16"
    grad_dtype: str = "bf16"
    seed: int = 0
    w_std: float = 0.02
    g_std: float = 1e-3
    outlier_frac: float = 0.0
    step: int = 1
    prior_moments: bool = False
    hp: tuple = (1e-3, 0.9, 0.999, 1e-8, 0.01)


def host_inputs(case: UnitCase):
    P = int(sum(int(np.prod(s, dtype=np.int64)) for s in case.shapes))
    w = synth.host_normal(1000 + case.seed, P, case.w_std)
    grads = []
    for r in range(case.R):
        g = synth.host_normal(2000 + case.seed + 101 * r, P, case.g_std)
        if case.outlier_frac:
            mask = np.random.default_rng(3000 + case.seed + 101 * r).random(P) < case.outlier_frac
            g[mask] *= np.float32(1e4)
        grads.append(synth.to_bf16_bits(g) if case.grad_dtype == "bf16" else g)
    return w, grads


def run_unit_case(case: UnitCase, w=None, grads=None, moments=None):
    """Pack, all-gather, reduce-scatter+AdamW, all-gather again: CUDA vs oracle."""
    if w is None:
        w, grads = host_inputs(case)
    O = oracle.layout(omode(case.mode), case.R, case.shapes)
    U = ShardedUnit(case.shapes, case.R, case.mode, case.param_dtype, case.grad_dtype)
    assert (U.P, U.S) == (O.full_numel, O.shard_numel)
    bf16 = case.param_dtype == "bf16"

    # a2: shard from full
    U.shard_from_full(to_dev(w))
    masters, p16 = oracle.pack(O, w, with_bf16=bf16)
    for r in range(case.R):
        assert_bits_equal(host(U.master[r]), masters[r], f"pack master[{r}]")
        if bf16:
            assert_bits_equal(host(U.param_shard[r]), p16[r], f"pack bf16[{r}]")

    # a3: all-gather + unflatten
    full = U.alloc_full()
    U.all_gather(full)
    want_full = oracle.all_gather(O, p16 if bf16 else masters)
    for d in range(case.R):
        assert_bits_equal(host(full[d]), want_full[d], f"all-gather full[{d}]")

    # a4-a6: reduce-scatter + AdamW
    if moments is None and case.prior_moments:
        wl = synth.Workload("case", case.seed, case.mode, case.R, (), case.param_dtype,
                            case.grad_dtype, case.w_std, case.g_std)
        moments = synth.host_moments(wl, 0, U.S)
    m = [np.zeros(U.S, np.float32) for _ in range(case.R)]
    v = [np.zeros(U.S, np.float32) for _ in range(case.R)]
    if moments is not None:
        m = [x.copy() for x in moments[0]]
        v = [x.copy() for x in moments[1]]
        for r in range(case.R):
            U.m[r].copy_(to_dev(m[r]))
            U.v[r].copy_(to_dev(v[r]))
    lr, b1, b2, eps, wd = case.hp
    gdev = [to_dev(g) for g in grads]
    gsh = [torch.zeros(U.S, dtype=torch.float32, device="cuda") for _ in range(case.R)]
    U.reduce_scatter_adamw(gdev, AdamWHP(lr, b1, b2, eps, wd), grad_shard_out=gsh,
                           step=case.step)
    want_g, want_p16 = oracle.rs_adamw(O, grads, masters, m, v,
                                       oracle.AdamWHP(lr, b1, b2, eps, wd), case.step,
                                       with_bf16=bf16)
    exact_master = 0
    for r in range(case.R):
        assert_bits_equal(host(gsh[r]), want_g[r], f"reduce-scatter shard[{r}]")
        gm = host(U.master[r])
        assert_master_close(gm, masters[r], f"master[{r}]")
        exact_master += int(np.sum(gm.view(np.uint32) == masters[r].view(np.uint32)))
        assert_moment_close(host(U.m[r]), m[r], f"m[{r}]")
        assert_moment_close(host(U.v[r]), v[r], f"v[{r}]")
        if bf16:
            assert_bf16_close(host(U.param_shard[r]), want_p16[r], f"bf16 shard[{r}]")

    # gather of the updated shards, against the oracle's gather of its own
    U.all_gather(full)
    want_full = oracle.all_gather(O, want_p16 if bf16 else masters)
    for d in range(case.R):
        got = host(full[d])
        if bf16:
            assert_bf16_close(got, want_full[d], f"gather after step full[{d}]")
        else:
            assert_master_close(got, want_full[d], f"gather after step full[{d}]")
    torch.cuda.synchronize()
    return {"P": U.P, "exact_master_fraction": exact_master / max(1, case.R * U.S)}


def run_overlap_case(case_rs: UnitCase, case_ag: UnitCase, seed_shift: int = 500):
    """The prefetch call: reduce-scatter + AdamW of one unit and all-gather
    of another, each compared with the oracle."""
    w_a, grads = host_inputs(case_rs)
    case_b = UnitCase(**{**case_ag.__dict__, "seed": case_ag.seed + seed_shift})
    w_b, _ = host_inputs(case_b)
    mk = lambda c: (oracle.layout(omode(c.mode), c.R, c.shapes),
                    ShardedUnit(c.shapes, c.R, c.mode, c.param_dtype, c.grad_dtype))
    Oa, Ua = mk(case_rs)
    Ob, Ub = mk(case_b)
    bf_a, bf_b = case_rs.param_dtype == "bf16", case_b.param_dtype == "bf16"
    Ua.shard_from_full(to_dev(w_a))
    Ub.shard_from_full(to_dev(w_b))
    masters_a, _ = oracle.pack(Oa, w_a, with_bf16=bf_a)
    masters_b, p16_b = oracle.pack(Ob, w_b, with_bf16=bf_b)
    m = [np.zeros(Ua.S, np.float32) for _ in range(case_rs.R)]
    v = [np.zeros(Ua.S, np.float32) for _ in range(case_rs.R)]
    lr, b1, b2, eps, wd = case_rs.hp
    full_b = Ub.alloc_full()
    gsh = [torch.zeros(Ua.S, dtype=torch.float32, device="cuda") for _ in range(case_rs.R)]
    Ua.reduce_scatter_adamw_and_gather([to_dev(g) for g in grads], AdamWHP(lr, b1, b2, eps, wd),
                                       Ub, full_b, grad_shard_out=gsh, step=case_rs.step)
    want_g, want_p16 = oracle.rs_adamw(Oa, grads, masters_a, m, v,
                                       oracle.AdamWHP(lr, b1, b2, eps, wd), case_rs.step,
                                       with_bf16=bf_a)
    want_full = oracle.all_gather(Ob, p16_b if bf_b else masters_b)
    for d in range(case_b.R):
        assert_bits_equal(host(full_b[d]), want_full[d], f"overlapped gather full[{d}]")
    for r in range(case_rs.R):
        assert_bits_equal(host(gsh[r]), want_g[r], f"overlapped reduce-scatter shard[{r}]")
        assert_master_close(host(Ua.master[r]), masters_a[r], f"overlapped master[{r}]")
        assert_moment_close(host(Ua.m[r]), m[r], f"overlapped m[{r}]")
        assert_moment_close(host(Ua.v[r]), v[r], f"overlapped v[{r}]")
        if bf_a:
            assert_bf16_close(host(Ua.param_shard[r]), want_p16[r], f"overlapped bf16[{r}]")
    torch.cuda.synchronize()


def run_accumulation_case(case: UnitCase, K: int):
    """K micro-batches: accumulate K-1 on the GPU, fuse the last into the
    reduce-scatter + AdamW; compare with the oracle accumulating all K and
    reduce-scattering the accumulators. Also checks that the unfused GPU path
    (accumulate all K, reduce-scatter fp32 accumulators) gives the same bits."""
    w, _ = host_inputs(case)
    micro = [host_inputs(UnitCase(**{**case.__dict__, "seed": case.seed + 17 * k}))[1]
             for k in range(K)]
    O = oracle.layout(omode(case.mode), case.R, case.shapes)
    U = ShardedUnit(case.shapes, case.R, case.mode, case.param_dtype, case.grad_dtype)
    bf16 = case.param_dtype == "bf16"
    U.shard_from_full(to_dev(w))
    masters, _ = oracle.pack(O, w, with_bf16=bf16)
    acc = U.alloc_accumulators()
    o_acc = [np.zeros(U.P, np.float32) for _ in range(case.R)]
    for k in range(K - 1):
        U.accumulate_grad([to_dev(g) for g in micro[k]], acc, first=(k == 0))
        oracle.accumulate(o_acc, micro[k], first=(k == 0))
    for r in range(case.R):
        if K > 1:
            assert_bits_equal(host(acc[r]), o_acc[r], f"accumulator[{r}]")
    oracle.accumulate(o_acc, micro[K - 1], first=(K == 1))
    lr, b1, b2, eps, wd = case.hp
    gsh = [torch.zeros(U.S, dtype=torch.float32, device="cuda") for _ in range(case.R)]
    last = [to_dev(g) for g in micro[K - 1]]
    if K == 1:
        for a in acc:
            a.zero_()
    U.reduce_scatter_adamw_accum(acc, last, AdamWHP(lr, b1, b2, eps, wd), grad_shard_out=gsh,
                                 step=case.step)
    m = [np.zeros(U.S, np.float32) for _ in range(case.R)]
    v = [np.zeros(U.S, np.float32) for _ in range(case.R)]
    want_g, want_p16 = oracle.rs_adamw(O, o_acc, masters, m, v,
                                       oracle.AdamWHP(lr, b1, b2, eps, wd), case.step,
                                       with_bf16=bf16)
    for r in range(case.R):
        assert_bits_equal(host(gsh[r]), want_g[r], f"accumulated reduce-scatter shard[{r}]")
        assert_master_close(host(U.master[r]), masters[r], f"accumulated master[{r}]")
        assert_moment_close(host(U.m[r]), m[r], f"accumulated m[{r}]")
        assert_moment_close(host(U.v[r]), v[r], f"accumulated v[{r}]")
        if bf16:
            assert_bf16_close(host(U.param_shard[r]), want_p16[r], f"accumulated bf16[{r}]")
    # unfused: accumulate the last micro-batch too, reduce-scatter the accumulators
    if K > 1:
        U.accumulate_grad(last, acc, first=False)
        F = ShardedUnit(case.shapes, case.R, case.mode, case.param_dtype, "f32")
        F.shard_from_full(to_dev(w))
        gsh2 = [torch.zeros(F.S, dtype=torch.float32, device="cuda") for _ in range(case.R)]
        F.reduce_scatter_adamw(acc, AdamWHP(lr, b1, b2, eps, wd), grad_shard_out=gsh2,
                               step=case.step)
        for r in range(case.R):
            assert torch.equal(gsh[r].view(torch.int32), gsh2[r].view(torch.int32))
            assert torch.equal(U.master[r].view(torch.int32), F.master[r].view(torch.int32))
    torch.cuda.synchronize()


def run_units_case(cases, step: int = 1, share_layout: bool = False):
    """Several units through the multi-unit calls (one launch where they fit):
    all-gather + unflatten of every unit, then reduce-scatter + AdamW of every
    unit, each unit compared with the oracle on its own inputs."""
    from fully_sharded_state_gb300 import all_gather_units, reduce_scatter_adamw_units
    c0 = cases[0]
    bf16 = c0.param_dtype == "bf16"
    units, Os, ws, gs = [], [], [], []
    for c in cases:
        w, grads = host_inputs(c)
        U = ShardedUnit(c.shapes, c.R, c.mode, c.param_dtype, c.grad_dtype)
        if share_layout and units:
            U.layout = units[0].layout  # one layout object serving several units
        U.shard_from_full(to_dev(w))
        units.append(U)
        Os.append(oracle.layout(omode(c.mode), c.R, c.shapes))
        ws.append(w)
        gs.append(grads)
    fulls = [U.alloc_full() for U in units]
    all_gather_units(units, fulls)
    packed = [oracle.pack(O, w, with_bf16=bf16) for O, w in zip(Os, ws)]
    for u, (O, (masters, p16)) in enumerate(zip(Os, packed)):
        want = oracle.all_gather(O, p16 if bf16 else masters)
        for d in range(c0.R):
            assert_bits_equal(host(fulls[u][d]), want[d], f"unit {u} full[{d}]")
    lr, b1, b2, eps, wd = c0.hp
    gsh = [[torch.zeros(U.S, dtype=torch.float32, device="cuda") for _ in range(c0.R)]
           for U in units]
    reduce_scatter_adamw_units(units, [[to_dev(g) for g in grads] for grads in gs],
                               AdamWHP(lr, b1, b2, eps, wd), grad_shard_outs=gsh, step=step)
    for u, (U, O, (masters, _)) in enumerate(zip(units, Os, packed)):
        m = [np.zeros(U.S, np.float32) for _ in range(c0.R)]
        v = [np.zeros(U.S, np.float32) for _ in range(c0.R)]
        want_g, want_p16 = oracle.rs_adamw(O, gs[u], masters, m, v,
                                           oracle.AdamWHP(lr, b1, b2, eps, wd), step,
                                           with_bf16=bf16)
        assert U.step == step
        for r in range(c0.R):
            assert_bits_equal(host(gsh[u][r]), want_g[r], f"unit {u} reduce-scatter[{r}]")
            assert_master_close(host(U.master[r]), masters[r], f"unit {u} master[{r}]")
            assert_moment_close(host(U.m[r]), m[r], f"unit {u} m[{r}]")
            assert_moment_close(host(U.v[r]), v[r], f"unit {u} v[{r}]")
            if bf16:
                assert_bf16_close(host(U.param_shard[r]), want_p16[r], f"unit {u} bf16[{r}]")
    torch.cuda.synchronize()
    return units
