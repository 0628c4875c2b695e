"""Host logic of bench.py without a GPU: the algorithmic byte counts, the
max-over-ranks timing across two gloo ranks, and the reference arm's line."""
import json
import os
import socket

import torch.multiprocessing as mp

import bench


def test_algorithmic_bytes():
    # four Llama-style blocks, R = 8, bf16: 42 bytes per parameter for the
    # fused reduce-scatter + AdamW, 18 for the all-gather
    P = 218_112_000
    assert bench.rs_adamw_bytes(P, 8) == 9_160_704_000
    assert bench.all_gather_bytes(P, 8) == 3_926_016_000
    # the 512/8/2048 block with its LayerNorm scales, R = 4
    P = 3_146_752
    assert bench.rs_adamw_bytes(P, 4) == 106_989_568
    assert bench.all_gather_bytes(P, 4) == 31_467_520
    # fp32 parameters and gradients: 4R + 24
    assert bench.rs_adamw_bytes(10, 8, grad_b=4, param_b=0) == 10 * (4 * 8 + 24)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    got = bench.max_over_ranks(10.0 + 3 * rank, world)
    out[rank] = got
    dist.destroy_process_group()


def test_rs_kernel_name_follows_the_staging_rule():
    from fully_sharded_state_gb300 import synth
    llama = synth.WORKLOADS["llama4"].unit_shapes(0)
    block = synth.WORKLOADS["block"].unit_shapes(0)
    # Llama unit: 106K tiles at R = 8, bf16 gradients
    assert bench.rs_kernel_name(llama, 8, 2, 152) == "rs_adamw_staged_kernel"
    assert bench.rs_kernel_name(llama, 4, 2, 152) == "rs_adamw_staged_kernel"
    assert bench.rs_kernel_name(llama, 2, 4, 152) == "rs_adamw_staged_kernel"
    # too few gradient bytes per element, or a stage over 32 KB, or R unknown
    # at compile time
    assert bench.rs_kernel_name(llama, 2, 2, 152) == "rs_adamw_kernel"
    assert bench.rs_kernel_name(llama, 8, 4, 152) == "rs_adamw_kernel"
    assert bench.rs_kernel_name(llama, 16, 2, 152) == "rs_adamw_kernel"
    # the 3.1M-parameter block: 1,536 tiles, under 32 per staged thread block
    assert bench.rs_kernel_name(block, 4, 2, 152) == "rs_adamw_kernel"
    # the bar: 32 tiles x 2 thread blocks x SMs
    assert bench.rs_kernel_name([(9728 * 2048,)], 4, 2, 152) == "rs_adamw_staged_kernel"
    assert bench.rs_kernel_name([(9724 * 2048,)], 4, 2, 152) == "rs_adamw_kernel"
    # 16 tiles when most rank pieces start off the 8-element grid: rows of
    # 2,999 x 1,001 put ranks 1-3 off it (5,864 tiles)
    assert bench.rs_kernel_name([(11996, 1001)], 4, 2, 152) == "rs_adamw_staged_kernel"
    assert bench.rs_kernel_name([(5996, 1001)], 4, 2, 152) == "rs_adamw_kernel"


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 13.0, 1: 13.0}


def test_reference_arm_line(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "0")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["value"] > 0


def test_reference_arm_other_ranks_do_nothing(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""
