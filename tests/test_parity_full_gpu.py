"""Full-size parity: Llama-style decoder blocks (hidden 4096, ffn 14336, GQA),
one FSDP unit per block, R = 8, bf16 parameters and gradients, through the
same library calls the benchmark times (no gradient-shard output).

Inputs come from the seeded device generator. The oracle computes sampled
outputs one by one: for all-gather, the owner slot of each sampled unit
element; for reduce-scatter + AdamW, the rank-ordered fp32 sum of the sampled
elements' R gradients and the AdamW step on their saved state. Samples are
uniform over the unit plus the first and last two elements of every rank
piece of every parameter. Properties that hold at any size are checked on
whole buffers."""
import numpy as np
import pytest
import torch

import oracle
from fully_sharded_state_gb300 import AdamWHP, ShardedUnit, synth
from parity import (assert_bf16_close, assert_bits_equal, assert_master_close,
                    assert_moment_close, host)

pytestmark = pytest.mark.gpu


def _sample(O, rng, n=40000):
    P = O.full_numel
    js = set(rng.integers(0, P, n).tolist())
    for i in range(len(O.shapes)):
        for r in range(O.R):
            s, c = O.rank_rows(i, r)
            if c:
                a = int(O.full_off[i] + s * O.inner[i])
                b = a + c * int(O.inner[i])
                js.update([a, a + 1, b - 2, b - 1])
    js.update([0, P - 1])
    return np.array(sorted(j for j in js if 0 <= j < P), np.int64)


def _at(bufs, rank, idx, dev):
    """Values of per-rank buffers at (rank[k], idx[k])."""
    out = None
    for r in np.unique(rank):
        sel = np.flatnonzero(rank == r)
        vals = host(bufs[r][torch.from_numpy(idx[sel]).to(dev)])
        if out is None:
            out = np.empty(rank.size, vals.dtype)
        out[sel] = vals
    return out


@pytest.mark.parametrize("u", [0, 3])
def test_llama_unit_full_size_sampled(cuda_lib, u):
    wl = synth.WORKLOADS["llama4"]
    dev = torch.device("cuda")
    shapes = wl.unit_shapes(u)
    U = ShardedUnit(shapes, wl.R, "per_param", "bf16", "bf16", names=[n for n, _ in wl.units[u]])
    O = oracle.layout(oracle.PER_PARAM, wl.R, shapes)
    assert (U.P, U.S) == (O.full_numel, O.shard_numel) == (218_112_000, 27_264_000)
    base = synth.seed("w", wl, u)
    for r in range(wl.R):
        U.param_shard[r].copy_(synth.device_normal(base + r, U.S, wl.w_std, dev, torch.bfloat16))
        U.master[r].copy_(synth.device_normal(base + 50 + r, U.S, wl.w_std, dev))
    ms, vs = synth.device_moments(wl, u, U.S, dev)
    for r in range(wl.R):
        U.m[r].copy_(ms[r])
        U.v[r].copy_(vs[r])
    del ms, vs
    grads = synth.device_grads(wl, u, dev)
    rng = np.random.default_rng(100 + u)
    js = _sample(O, rng)
    rank, idx = oracle.owner(O, js)
    jt = torch.from_numpy(js).to(dev)

    # all-gather + unflatten
    full = U.alloc_full()
    U.all_gather(full)
    want = _at(U.param_shard, rank, idx, dev)
    for d in range(wl.R):
        assert_bits_equal(host(full[d][jt]), want, f"full[{d}] at samples")
    for d in range(1, wl.R):  # every destination receives the same bytes
        assert torch.equal(full[d].view(torch.int16), full[0].view(torch.int16))
    views = U.unflatten(full[0])
    assert tuple(views["W_down"].shape) == (4096, 14336)
    del full

    # reduce-scatter + AdamW (step 3 with prior moments)
    hp = AdamWHP(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay)
    ohp = oracle.AdamWHP(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay)
    g_s = [host(grads[q][jt]) for q in range(wl.R)]
    w_s, m_s, v_s = (_at(b, rank, idx, dev) for b in (U.master, U.m, U.v))
    U.reduce_scatter_adamw(grads, hp, step=3)
    torch.cuda.synchronize()
    gs = oracle.sum_ranks(g_s)
    w_o, m_o, v_o = w_s.copy(), m_s.copy(), v_s.copy()
    oracle.adamw(gs, w_o, m_o, v_o, ohp, 3)
    assert_master_close(_at(U.master, rank, idx, dev), w_o)
    assert_moment_close(_at(U.m, rank, idx, dev), m_o, "m")
    assert_moment_close(_at(U.v, rank, idx, dev), v_o, "v")
    assert_bf16_close(_at(U.param_shard, rank, idx, dev), oracle.f32_to_bf16(w_o))
    # the bf16 shard is the rounding of the new master everywhere
    for r in range(wl.R):
        assert torch.equal(U.param_shard[r].view(torch.int16),
                           U.master[r].to(torch.bfloat16).view(torch.int16))

    # the reduced gradient itself, bit-exact at the samples
    gsh = [torch.zeros(U.S, dtype=torch.float32, device=dev) for _ in range(wl.R)]
    U.reduce_scatter_adamw(grads, hp, grad_shard_out=gsh, step=4)
    assert_bits_equal(_at(gsh, rank, idx, dev), gs, "reduce-scatter shard at samples")
    torch.cuda.synchronize()


@pytest.mark.parametrize("R,P", [
    (2, (1 << 31) + 4097),   # the register reduce-scatter (bf16, R = 2)
    (4, (1 << 31) + 32768),  # the staged one; rank 3's aligned piece straddles 2^31
])
def test_unit_past_two_to_the_31_elements(cuda_lib, R, P):
    """A FlatParameter unit of just over 2^31 bf16 elements (about 47-64 GB
    on the device): element offsets and tile indices pass 2^31, and byte
    offsets pass 4 GB, so the 64-bit index paths run, including the staged
    reduce-scatter's bulk-copy addresses at R = 4. Samples cluster around
    2^31, the rank boundaries and the end of the unit."""
    dev = torch.device("cuda")
    shapes = [(P,)]
    U = ShardedUnit(shapes, R, "flat", "bf16", "bf16")
    O = oracle.layout(oracle.FLAT, R, shapes)
    assert (U.P, U.S) == (O.full_numel, O.shard_numel)
    for r in range(R):
        U.param_shard[r].copy_(synth.device_normal(900 + r, U.S, 0.02, dev, torch.bfloat16))
        U.master[r].copy_(synth.device_normal(910 + r, U.S, 0.02, dev))
        U.m[r].copy_(synth.device_normal(920 + r, U.S, 1e-4, dev))
        z = synth.device_normal(930 + r, U.S, 1e-3, dev)
        U.v[r].copy_(z.mul_(z).mul_(1e-3))
        del z
    rng = np.random.default_rng(7)
    js = set()
    for c in [0, 1 << 31, P - 1] + [r * U.S + o for r in range(1, R) for o in (-1, 0)]:
        js.update(range(max(0, c - 40), min(P, c + 40)))
    js.update(rng.integers(0, P, 20000).tolist())
    js = np.array(sorted(js), np.int64)
    rank, idx = oracle.owner(O, js)
    jt = torch.from_numpy(js).to(dev)

    full = U.alloc_full()
    U.all_gather(full)
    want = _at(U.param_shard, rank, idx, dev)
    for d in range(R):
        assert_bits_equal(host(full[d][jt]), want, f"full[{d}] past 2^31")
    del full
    grads = [synth.device_normal(940 + q, P, 1e-3, dev, torch.bfloat16) for q in range(R)]
    hp = AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01)
    ohp = oracle.AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01)
    g_s = [host(grads[q][jt]) for q in range(R)]
    w_s, m_s, v_s = (_at(b, rank, idx, dev) for b in (U.master, U.m, U.v))
    U.reduce_scatter_adamw(grads, hp, step=2)
    torch.cuda.synchronize()
    gs = oracle.sum_ranks(g_s)
    w_o, m_o, v_o = w_s.copy(), m_s.copy(), v_s.copy()
    oracle.adamw(gs, w_o, m_o, v_o, ohp, 2)
    assert_master_close(_at(U.master, rank, idx, dev), w_o)
    assert_moment_close(_at(U.m, rank, idx, dev), m_o, "m")
    assert_moment_close(_at(U.v, rank, idx, dev), v_o, "v")
    assert_bf16_close(_at(U.param_shard, rank, idx, dev), oracle.f32_to_bf16(w_o))
    torch.cuda.synchronize()


def test_llama_unit_whole_vs_oracle(cuda_lib):
    """One whole Llama-style unit (218,112,000 parameters, R = 8, bf16
    parameters and gradients) through the calls the benchmark times, every
    output element compared with the oracle on the same host-generated
    inputs: pack (bit-exact), all 8 gather destinations (bit-exact), the fp32
    reduce-scatter shard (bit-exact), master/m/v after a step-3 update from
    prior moments (1e-5 bounds), the bf16 shard (1 ulp), and the gather of
    the updated shards."""
    wl = synth.WORKLOADS["llama4"]
    u = 1
    shapes = wl.unit_shapes(u)
    R = wl.R
    dev = torch.device("cuda")
    O = oracle.layout(oracle.PER_PARAM, R, shapes)
    U = ShardedUnit(shapes, R, "per_param", "bf16", "bf16", names=[n for n, _ in wl.units[u]])
    assert (U.P, U.S) == (O.full_numel, O.shard_numel) == (218_112_000, 27_264_000)

    # a2: shard from full
    w = synth.host_weights(wl, u)
    U.shard_from_full(torch.from_numpy(w).to(dev))
    masters, p16 = oracle.pack(O, w, with_bf16=True)
    del w
    for r in range(R):
        assert_bits_equal(host(U.master[r]), masters[r], f"pack master[{r}]")
        assert_bits_equal(host(U.param_shard[r]), p16[r], f"pack bf16[{r}]")

    # a3: all-gather + unflatten, every destination, every element
    full = U.alloc_full()
    U.all_gather(full)
    want = oracle.all_gather(O, p16)
    for d in range(R):
        assert_bits_equal(host(full[d]), want[d], f"all-gather full[{d}]")
    del want

    # a4-a6: reduce-scatter + AdamW at step 3 from prior moments
    ms, vs = synth.host_moments(wl, u, U.S)
    for r in range(R):
        U.m[r].copy_(torch.from_numpy(ms[r]))
        U.v[r].copy_(torch.from_numpy(vs[r]))
    grads = synth.host_grads(wl, u)
    gdev = [torch.from_numpy(g.view(np.int16)).to(dev).view(torch.bfloat16) for g in grads]
    gsh = [torch.empty(U.S, dtype=torch.float32, device=dev) for _ in range(R)]
    hp = AdamWHP(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay)
    U.reduce_scatter_adamw(gdev, hp, grad_shard_out=gsh, step=3)
    del gdev
    want_g, want_p16 = oracle.rs_adamw(O, grads, masters, ms, vs,
                                       oracle.AdamWHP(wl.lr, wl.betas[0], wl.betas[1], wl.eps,
                                                      wl.weight_decay), 3, with_bf16=True)
    del grads
    for r in range(R):
        n = O.rank_numel(r)  # the reduce-scatter writes owned elements only
        got_g = host(gsh[r])
        for i in range(len(shapes)):
            s, c = O.rank_rows(i, r)
            a = int(O.shard_off[i])
            b = a + c * int(O.inner[i])
            assert_bits_equal(got_g[a:b], want_g[r][a:b], f"reduce-scatter shard[{r}] param {i}")
        assert n > 0
        assert_master_close(host(U.master[r]), masters[r], f"master[{r}]")
        assert_moment_close(host(U.m[r]), ms[r], f"m[{r}]")
        assert_moment_close(host(U.v[r]), vs[r], f"v[{r}]")
        assert_bf16_close(host(U.param_shard[r]), want_p16[r], f"bf16 shard[{r}]")

    # the gather of the updated shards
    U.all_gather(full)
    want = oracle.all_gather(O, want_p16)
    for d in range(R):
        assert_bf16_close(host(full[d]), want[d], f"gather after the step full[{d}]")
    torch.cuda.synchronize()
