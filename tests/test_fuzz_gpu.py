"""Seeded random units through the CUDA path, each compared element by element
with the oracle: random layout mode (FSDP1 / FSDP2 / ZeRO-3), parameter and
gradient dtypes, R from 1 to 12, ragged shapes (empty parameters, rows fewer
than ranks, odd row widths), optimizer step and prior moments. Also random
prefetch and accumulation calls, and two host threads driving the library on
two streams at once."""
import threading

import numpy as np
import pytest
import torch

from parity import UnitCase, run_accumulation_case, run_overlap_case, run_unit_case

pytestmark = pytest.mark.gpu


def _random_case(rng, seed):
    n = int(rng.integers(1, 7))
    shapes = []
    for _ in range(n):
        nd = int(rng.integers(1, 4))
        d0 = int(rng.choice([0, 1, 2, 3, 5, 7, 31, 127, 513, 1000, 2049, 3001]))
        rest = [int(rng.choice([1, 3, 8, 33, 64, 127])) for _ in range(nd - 1)]
        shapes.append(tuple([d0] + rest))
    return UnitCase(shapes=shapes, R=int(rng.integers(1, 13)),
                    mode=str(rng.choice(["per_param", "flat", "zero3"])),
                    param_dtype=str(rng.choice(["bf16", "f32"])),
                    grad_dtype=str(rng.choice(["bf16", "f32"])),
                    seed=seed, g_std=float(rng.choice([1e-3, 1.0])),
                    outlier_frac=float(rng.choice([0.0, 0.01])),
                    step=int(rng.integers(1, 5)), prior_moments=bool(rng.integers(0, 2)))


@pytest.mark.parametrize("k", range(40))
def test_random_unit(cuda_lib, k):
    rng = np.random.default_rng(1000 + k)
    run_unit_case(_random_case(rng, 600 + k))


@pytest.mark.parametrize("k", range(8))
def test_random_prefetch(cuda_lib, k):
    rng = np.random.default_rng(2000 + k)
    a = _random_case(rng, 700 + k)
    b = _random_case(rng, 800 + k)
    if sum(int(np.prod(s)) for s in a.shapes) == 0:
        a.shapes = a.shapes + [(5, 3)]
    run_overlap_case(a, b)


@pytest.mark.parametrize("k", range(8))
def test_random_accumulation(cuda_lib, k):
    rng = np.random.default_rng(3000 + k)
    run_accumulation_case(_random_case(rng, 900 + k), int(rng.integers(1, 5)))


def test_two_threads_two_streams(cuda_lib):
    """Layouts and launches from two host threads at once (the library keeps
    no per-call state outside the caller's arguments and a locked device
    cache)."""
    from fully_sharded_state_gb300 import AdamWHP, ShardedUnit
    hp = AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01)
    errors = []

    def work(tid):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                U = ShardedUnit([(1000 + tid, 64), (77, 3)], R=4 + tid)
                w = torch.randn(U.P, device="cuda")
                g = [torch.randn(U.P, device="cuda").to(torch.bfloat16) for _ in range(U.R)]
                U.shard_from_full(w, stream=s)
                full = U.alloc_full()
                for _ in range(20):
                    U.all_gather(full, stream=s)
                    U.reduce_scatter_adamw(g, hp, stream=s)
                U.all_gather(full, stream=s)
            s.synchronize()
            for d in range(1, U.R):
                assert torch.equal(full[d].view(torch.int16), full[0].view(torch.int16))
        except Exception as e:  # surfaced to the main thread
            errors.append(e)

    ts = [threading.Thread(target=work, args=(t,)) for t in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors


def test_two_threads_staged_units_match_a_serial_run(cuda_lib):
    """Two host threads drive units large enough for the staged
    reduce-scatter (21M parameters; R = 8 and R = 4, so two different staged
    kernels) on their own streams at once, five steps each; every buffer
    must equal a serial run of the same steps bit for bit."""
    from fully_sharded_state_gb300 import AdamWHP, ShardedUnit, synth
    hp = AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01)
    shapes = [(4096, 4096), (1024, 4096), (4096,)]
    dev = torch.device("cuda")

    def run(R, stream):
        with torch.cuda.stream(stream):
            U = ShardedUnit(shapes, R)
            U.shard_from_full(synth.device_normal(10 + R, U.P, 0.02, dev), stream=stream)
            g = [synth.device_normal(20 + R + r, U.P, 1e-3, dev, torch.bfloat16)
                 for r in range(R)]
            full = U.alloc_full()
            for _ in range(5):
                U.all_gather(full, stream=stream)
                U.reduce_scatter_adamw(g, hp, stream=stream)
            U.all_gather(full, stream=stream)
        stream.synchronize()
        return [t.clone() for t in U.master + U.m + U.v + U.param_shard + full]

    got, errors = {}, []

    def work(R):
        try:
            got[R] = run(R, torch.cuda.Stream())
        except Exception as e:  # surfaced to the main thread
            errors.append(e)

    ts = [threading.Thread(target=work, args=(R,)) for R in (8, 4)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    bits = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)
    for R in (8, 4):
        want = run(R, torch.cuda.current_stream())
        for a, b in zip(got[R], want):
            assert torch.equal(bits(a), bits(b))


@pytest.mark.parametrize("k", range(12))
def test_random_units_per_call(cuda_lib, k):
    """Random groups of units through the multi-unit calls: 1 to 24 units
    sharing R and dtypes, each with its own shapes and layout mode, so the
    launches split by segment count and by pointer count; every unit is
    compared with the oracle."""
    from parity import run_units_case
    rng = np.random.default_rng(4000 + k)
    first = _random_case(rng, 1000 + k)
    cases = [first]
    for u in range(int(rng.integers(0, 24))):
        c = _random_case(rng, 1100 + 37 * k + u)
        c.R, c.param_dtype, c.grad_dtype = first.R, first.param_dtype, first.grad_dtype
        c.hp = first.hp
        cases.append(c)
    run_units_case(cases, step=int(rng.integers(1, 4)))
