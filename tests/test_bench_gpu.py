"""bench.py end to end on the GPU, on its small one-unit workload: the JSON
line carries every key of the benchmark contract with sane values."""
import json

import pytest

import bench

pytestmark = pytest.mark.gpu


def test_bench_line_contract(cuda_lib, capsys):
    bench.main(["--workload", "llama_attn", "--steps", "5", "--warmup", "3", "--no-configs",
                "--no-cpu-baseline"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "clocks", "gpu_launches", "e2e"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 5 and line["warmup"] >= 3
    assert line["value"] > 0 and line["gpu_launches"] == 5 * 2
    roof = line["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["bound"] == "hbm" and roof["achieved"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    # the host link's own rate over the same buffers, just before and after
    assert len(e2e["h2d_link_GBps_before_after"]) == 2
    assert all(x > 0 for x in e2e["h2d_link_GBps_before_after"])
    assert "workload" in line["config"]
    z1 = line["zero1"]
    assert z1["step_ms_per_unit"] > z1["fsdp_step_ms_per_unit"] > 0
    for entry in (line["roofline_all_gather"], line["ddp_all_reduce"], line["pack"],
                  z1["adamw_from_reduced"], *line["grad_accumulation"].values()):
        assert entry["achieved"] > 0
        assert entry["frac_of_nominal"] < entry["frac"]
    ceil = line["ceilings"]
    for key in ("write_only_x_R_gbs", "device_copy_x_R_gbs", "h2d_pinned_gbs", "d2h_pinned_gbs"):
        assert ceil[key] > 0, key
    assert "frac_of_write_ceiling" in roof
    # the step allocates nothing beyond the FSDP2 page's peak-memory terms
    for sched in ("in_order", "prefetch"):
        mem = line["peak_memory"][sched]
        assert abs(mem["measured_bytes"] - mem["formula_bytes"]) <= 65536, mem
    assert line["peak_memory"]["prefetch"]["M_prefetch"] > 0


def test_peak_memory_matches_the_pages_formula(cuda_lib):
    """Peak device memory of a step of twelve 512/8/2048 blocks (R = 4),
    in order and with prefetch, equals the FSDP2 page's §01 formula as the
    oracle states it: the peak of the bytes requested from the allocator
    (its own block rounding left out) equals the formula to within 64 KB."""
    import torch
    from fractions import Fraction

    from fully_sharded_state_gb300 import AdamWHP, synth
    from oracle import formulas

    wl = synth.WORKLOADS["block12_flat"]
    shapes = [wl.unit_shapes(u) for u in range(len(wl.units))]
    got = bench.peak_memory(torch, torch.device("cuda"), shapes, wl.R, "per_param",
                            AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01))
    P = wl.unit_numel(0)
    R = wl.R
    import oracle
    S = oracle.layout(oracle.PER_PARAM, R, shapes[0]).shard_numel
    # sharded state: bf16 shard + fp32 master (b_w = 6), no stored gradient
    # shard (b_g = 0), AdamW m and v (b_o = 8), for R ranks over 12 units
    m_shard = 12 * R * formulas.shard_state_bytes(S * R, 6, 0, 8, R)
    full_unit = R * P * 2
    for sched, prefetch in (("in_order", 0), ("prefetch", full_unit)):
        want = formulas.peak_bytes(m_shard, full_unit, prefetch, activations=0, temp=full_unit)
        assert want == Fraction(got[sched]["formula_bytes"])
        assert abs(got[sched]["measured_bytes"] - want) <= 65536, (sched, got[sched])


@pytest.mark.parametrize("shapes,R,gdt", [
    ([(4096, 4096), (1024, 4096), (4096,)], 8, "bf16"),  # staged
    ([(6000, 4097)], 4, "f32"),                           # staged, fp32 gradients
    ([(11996, 1001)], 4, "bf16"),                         # staged from 16 tiles a CTA:
                                                          # 3 of 4 rank pieces misaligned
    ([(512, 512), (512,)], 4, "bf16"),                    # too few tiles: register
    ([(6000, 4097)], 2, "bf16"),                          # 4 gradient bytes: register
    ([(6000, 4097)], 8, "f32"),                           # a 64 KB stage: register
])
def test_rs_kernel_name_matches_the_launched_kernel(cuda_lib, shapes, R, gdt):
    """The kernel bench.py names in its roofline is the one the library
    launches: the reduce-scatter runs under torch.profiler (CUPTI sees every
    kernel in the process) and the recorded name must match."""
    import torch
    from torch.profiler import ProfilerActivity, profile

    from fully_sharded_state_gb300 import AdamWHP, ShardedUnit

    U = ShardedUnit(shapes, R, "per_param", "bf16", gdt)
    U.shard_from_full(torch.randn(U.P, device="cuda") * 0.02)
    grads = U.alloc_grads()
    for g in grads:
        g.normal_(0, 1e-3)
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]):  # the first session starts CUPTI
        torch.zeros(1, device="cuda").add_(1)
        torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        U.reduce_scatter_adamw(grads, AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01))
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if "rs_adamw" in e.name]
    assert names, "the profiler recorded no reduce-scatter kernel"
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    want = bench.rs_kernel_name(U.shapes, R, 2 if gdt == "bf16" else 4, sms)
    assert any(want + "<" in n for n in names), (want, names)

