"""The OpenMP build of the oracle (the CPU baseline's multi-core figure)
gives the same bits as the plain single-thread build: its directives only
split element loops over threads, so every element's arithmetic is the same.
Checked on the ragged fp32 workload (R = 8, outliers) and the 512/8/2048
block (bf16, R = 4), for the all-gather, the fused reduce-scatter + AdamW from
prior moments, the all-reduce and the accumulation."""
import os

import numpy as np
import pytest

import oracle
from fully_sharded_state_gb300 import synth


def _run(wl, lib_path):
    with oracle.using(lib_path):
        u = 0
        shapes = wl.unit_shapes(u)
        bf16 = wl.param_dtype == "bf16"
        O = oracle.layout(oracle.FLAT if wl.mode == "flat" else oracle.PER_PARAM, wl.R, shapes)
        masters, p16 = oracle.pack(O, synth.host_weights(wl, u), with_bf16=bf16)
        full = oracle.all_gather(O, p16 if bf16 else masters)
        grads = synth.host_grads(wl, u)
        m, v = synth.host_moments(wl, u, O.shard_numel)
        hp = oracle.AdamWHP(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay)
        gsh, p16b = oracle.rs_adamw(O, grads, masters, m, v, hp, 4, with_bf16=bf16)
        ar = oracle.all_reduce(grads, out_bf16=False)
        acc = [np.zeros(O.full_numel, np.float32) for _ in range(wl.R)]
        oracle.accumulate(acc, grads, first=True)
        oracle.accumulate(acc, grads, first=False)
    out = full + gsh + masters + m + v + ar + acc + (p16b or [])
    return [np.ascontiguousarray(x).view(np.uint8) for x in out]


@pytest.mark.parametrize("name", ["ragged", "block"])
def test_openmp_build_is_bit_identical(name, monkeypatch):
    monkeypatch.setenv("OMP_NUM_THREADS", str(max(2, min(8, os.cpu_count() or 2))))
    wl = synth.WORKLOADS[name]
    plain = _run(wl, oracle.build())
    omp = _run(wl, oracle.build(openmp=True))
    assert len(plain) == len(omp)
    for k, (a, b) in enumerate(zip(plain, omp)):
        assert np.array_equal(a, b), f"output {k} differs between the builds"
