"""bench.py end to end on the GPU, on its small one-unit workload: the JSON
line carries every key of the benchmark contract with sane values."""
import json

import pytest

import bench

pytestmark = pytest.mark.gpu


def test_bench_line_contract(cuda_lib, capsys):
    bench.main(["--workload", "llama_attn", "--steps", "5", "--warmup", "3", "--no-small",
                "--no-cpu-baseline", "--e2e-steps", "2"])
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
    assert "workload" in line["config"]
    for entry in (line["roofline_all_gather"], line["ddp_all_reduce"], line["pack"],
                  *line["grad_accumulation"].values()):
        assert entry["achieved"] > 0
