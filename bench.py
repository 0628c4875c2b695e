"""Benchmark of the FSDP per-unit shard engine on GB300.

One step = one pass of the hot path over every FSDP unit of the workload:
for each unit, the parameter all-gather + unflatten (R full outputs) and the
fused fixed-order fp32 reduce-scatter + sharded AdamW. The layout is built
once; the shards are packed once before timing.

Workload (default): four Llama-style decoder blocks (hidden 4096, ffn 14336,
GQA with 1024-wide K/V; 218,112,000 parameters each), one FSDP2 unit per
block, R = 8 virtual ranks in this GPU's HBM, bf16 parameters and gradients,
fp32 master/m/v, seeded synthetic data. Each launch streams >= 3.9 GB, far
more than the 129 MB L2, so no L2 flush is needed between iterations.

value = algorithmic HBM bytes of all kernels of a step / device time of a
step, in GB/s, summed over GPUs (replicas) for N > 1.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama4|llama_attn] [--no-e2e] [--no-cpu-baseline]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

METRIC = "fused reduce-scatter+AdamW and all-gather HBM GB/s per FSDP unit; % of HBM peak"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- workload --

def workload_units(name: str):
    """(description, list of units (list of (name, shape)), R, dtypes)."""
    from fully_sharded_state_gb300 import synth
    wl = synth.WORKLOADS["llama4"]
    if name == "llama4":
        units = [list(u) for u in wl.units]
        desc = ("4 Llama-style decoder blocks (hidden 4096, ffn 14336, GQA kv 1024), one FSDP2 "
                "per-parameter unit per block (218,112,000 params), R=8 virtual ranks, bf16 "
                "params/grads, fp32 master/m/v")
    elif name == "llama_attn":
        # the attention part of one block: a smaller case for profiler captures
        units = [[p for p in wl.units[0] if p[0] in ("W_q", "W_k", "W_v", "W_o", "attn_norm")]]
        desc = ("attention weights of one Llama-style block (W_q, W_k, W_v, W_o, norm; "
                "41,947,136 params), FSDP2 unit, R=8, bf16 params/grads, fp32 state")
    else:
        raise SystemExit(f"unknown workload {name}")
    return desc, units, wl


def rs_adamw_bytes(P: int, R: int, grad_b: int = 2, param_b: int = 2) -> int:
    """Algorithmic bytes of one reduce-scatter + AdamW launch over a unit of P
    elements: R full gradients read, master/m/v read and written (24 B), the
    bf16 parameter shard written."""
    return P * (R * grad_b + 24 + param_b)


def all_gather_bytes(P: int, R: int, param_b: int = 2) -> int:
    """Algorithmic bytes of one all-gather: every shard element read once and
    written to R full outputs."""
    return P * param_b * (1 + R)


# ------------------------------------------------------------------ helpers --

def measured_peak():
    path = os.path.join(HERE, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


def kernel_source_hash() -> str:
    p = os.path.join(HERE, "fully_sharded_state_gb300", "csrc", "fsdp_kernels.cu")
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(HERE, "profiles", "dram_traffic__engine_kernels.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel]
        if e.get("kernel_source_sha256_16") != kernel_source_hash():
            return None
        if e.get("workload") == workload:
            return float(e["dram_bytes_per_launch"])
        return float(e["dram_bytes_per_launch_scaled"][workload])
    except Exception:
        return None


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.seek(0)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.out.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup(n_gpus: int):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (the job's time is its slowest rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------- CPU oracle --

class OracleSample:
    """A bounded sample of the workload for the CPU oracle (as it stands): the
    first `n_params` parameters of one block (W_q, W_k by default) as one
    FSDP2 unit, R = 8. Inputs are generated once; each run() times the
    oracle's all-gather of the bf16 shards and its reduce-scatter + AdamW."""

    def __init__(self, wl, n_params: int = 2):
        import oracle
        from fully_sharded_state_gb300 import synth
        self.oracle = oracle
        shapes = [s for _, s in wl.units[0][:n_params]]
        names = [n for n, _ in wl.units[0][:n_params]]
        self.L = L = oracle.layout(oracle.PER_PARAM, wl.R, shapes)
        P = L.full_numel
        w = synth.host_normal(7, P, wl.w_std)
        self.masters, self.p16 = oracle.pack(L, w, with_bf16=True)
        self.grads = [synth.to_bf16_bits(synth.host_normal(8 + q, P, wl.g_std))
                      for q in range(wl.R)]
        self.m = [np.zeros(L.shard_numel, np.float32) for _ in range(wl.R)]
        self.v = [np.zeros(L.shard_numel, np.float32) for _ in range(wl.R)]
        self.hp = oracle.AdamWHP(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay)
        self.t = 0
        self.nbytes = all_gather_bytes(P, wl.R) + rs_adamw_bytes(P, wl.R)
        self.desc = (f"{'+'.join(names)} of one block ({P:,} params), R={wl.R}: oracle "
                     "all-gather + reduce-scatter/AdamW, single thread")

    def run(self) -> float:
        self.t += 1
        t0 = time.perf_counter()
        self.oracle.all_gather(self.L, self.p16)
        _, self.p16 = self.oracle.rs_adamw(self.L, self.grads, self.masters, self.m, self.v,
                                           self.hp, self.t, with_bf16=True)
        return time.perf_counter() - t0


def host_cpu() -> str:
    """The host CPU's model as /proc/cpuinfo names it (Arm parts report an
    implementer/part pair instead of a model name)."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return "unknown"
    for key in ("model name", "Model name", "CPU part"):
        for line in info:
            if line.startswith(key):
                return f"{key}: {line.split(':', 1)[1].strip()}"
    return "unknown"


def cpu_baseline(wl, target_s: float = 10.0):
    smp = OracleSample(wl)
    dt = smp.run()
    reps = max(1, min(30, int(target_s / max(dt, 1e-3))))
    total_t = dt + sum(smp.run() for _ in range(reps - 1))
    return {"value": round(reps * smp.nbytes / total_t / 1e9, 4), "unit": UNIT, "cores": 1,
            "kind": "oracle", "sample": f"{reps} runs of {smp.desc}",
            "seconds": round(total_t, 2), "host_cores_available": os.cpu_count(),
            "host_cpu": host_cpu()}


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    desc, units, wl = workload_units(args.workload)
    smp = OracleSample(wl)
    for _ in range(args.warmup):
        smp.run()
    t_sum = sum(smp.run() for _ in range(args.steps))
    value = args.steps * smp.nbytes / t_sum / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t_sum / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": desc, "reference": "CPU oracle (plain C, one thread); each "
                       "step is a bounded sample of the workload"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1,
                             "kind": "oracle", "sample": smp.desc},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm --

def run_ours(args):
    import torch
    from fully_sharded_state_gb300 import AdamWHP, ShardedUnit, build, capi, synth

    rank, world, local = dist_setup(args.gpus)
    build.build()
    capi.load()
    dev = torch.device("cuda", local)
    desc, units_spec, wl = workload_units(args.workload)
    R = wl.R
    hp = AdamWHP(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay)

    units, grads, pack_ms = [], [], []
    for u, spec in enumerate(units_spec):
        U = ShardedUnit([s for _, s in spec], R, "per_param", "bf16", "bf16", device=dev,
                        names=[n for n, _ in spec])
        w_full = synth.device_normal(synth.seed("w", wl, u), U.P, wl.w_std, dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        U.shard_from_full(w_full)
        b.record()
        b.synchronize()
        pack_ms.append(a.elapsed_time(b))
        del w_full
        units.append(U)
        grads.append([synth.device_normal(synth.seed("g", wl, u, r), U.P, wl.g_std, dev,
                                          torch.bfloat16) for r in range(R)])
    P_max = max(U.P for U in units)
    full = [torch.empty(P_max, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    stream = torch.cuda.current_stream(dev)

    ag_bytes = sum(all_gather_bytes(U.P, R) for U in units)
    rs_bytes = sum(rs_adamw_bytes(U.P, R) for U in units)
    step_bytes = ag_bytes + rs_bytes

    def fulls(U):
        return [f[:U.P] for f in full]

    def one_step(ev=None):
        for k, U in enumerate(units):
            if ev is not None:
                ev[k][0].record(stream)
            U.all_gather(fulls(U), stream=stream)
            if ev is not None:
                ev[k][1].record(stream)
            U.reduce_scatter_adamw(grads[k], hp, stream=stream)
            if ev is not None:
                ev[k][2].record(stream)

    for _ in range(max(3, args.warmup)):
        one_step()
    torch.cuda.synchronize(dev)

    # timed region: K steps, bracketed by barrier + synchronize
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    kev = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in units]
           for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize(dev)
        ev_start.record(stream)
        for s in range(args.steps):
            one_step(kev[s])
        ev_end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    elapsed_ms = ev_start.elapsed_time(ev_end)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    ag_ms = [kev[s][k][0].elapsed_time(kev[s][k][1]) for s in range(args.steps)
             for k in range(len(units))]
    rs_ms = [kev[s][k][1].elapsed_time(kev[s][k][2]) for s in range(args.steps)
             for k in range(len(units))]
    launches = args.steps * len(units) * 2

    peak, peak_src = measured_peak()
    ms_step = elapsed_ms / args.steps
    value = world * step_bytes / (ms_step * 1e-3) / 1e9

    def entry(kernel, nbytes, ms, traffic_key):
        """Roofline record of one kernel: algorithmic bytes per launch over its
        mean CUDA-event launch time, against the measured HBM peak."""
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"kernel": kernel, "bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                "unit": "GB/s", "frac": round(gbs / peak, 4), "peak_source": peak_src,
                "algorithmic_bytes_per_launch": int(nbytes), "avg_launch_ms": round(ms, 4),
                "traffic": profiled_traffic(traffic_key, args.workload) if traffic_key else None}

    def timed_launches(fn, n=20):
        for _ in range(3):
            fn()
        ms = []
        for _ in range(n):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return statistics.mean(ms)

    roofline = entry("rs_adamw_kernel (fused reduce-scatter + AdamW)", rs_bytes / len(units),
                     statistics.mean(rs_ms), "rs_adamw")
    roofline_ag = entry("all_gather_kernel (all-gather + unflatten)", ag_bytes / len(units),
                        statistics.mean(ag_ms), "all_gather")

    # DDP's collective on the same unit, for comparison: all-reduce of the R
    # bf16 gradients into R fp32 full outputs (reduce dtype fp32)
    U0 = units[0]
    ar_out = [torch.empty(U0.P, dtype=torch.float32, device=dev) for _ in range(R)]
    ar_ms = timed_launches(lambda: U0.all_reduce(grads[0], ar_out, "f32", stream=stream))
    del ar_out
    ddp = entry("all_reduce_kernel (DDP all-reduce: bf16 grads -> fp32 outputs)",
                R * U0.P * (2 + 4), ar_ms, "all_reduce")

    # gradient accumulation on the same unit: one more micro-batch added into
    # the fp32 accumulators, and the last micro-batch fused into the step
    acc = U0.alloc_accumulators()
    U0.accumulate_grad(grads[0], acc, first=True, stream=stream)
    acc_ms = timed_launches(lambda: U0.accumulate_grad(grads[0], acc, first=False, stream=stream))
    rsacc_ms = timed_launches(lambda: U0.reduce_scatter_adamw_accum(acc, grads[0], hp,
                                                                     stream=stream))
    del acc
    accumulation = {
        "accumulate": entry("accumulate_kernel (acc += bf16 micro-batch grads, R ranks)",
                            R * U0.P * (4 + 2 + 4), acc_ms, "accumulate"),
        "rs_adamw_accum": entry("rs_adamw_kernel with accumulators (last micro-batch fused "
                                "into reduce-scatter + AdamW)",
                                U0.P * (R * (4 + 2) + 24 + 2), rsacc_ms, "rs_adamw_accum")}
    pack = entry("pack_kernel (shard from full: fp32 master + bf16 shard; set-up, untimed "
                 "step)", U0.P * 4 + R * U0.S * (4 + 2), statistics.mean(pack_ms[1:] or pack_ms),
                 "pack")

    small = None if args.no_small else small_configs(dev, hp)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, units, grads, full, hp, stream, dev, world, step_bytes)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": max(3, args.warmup),
                "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": desc, "units": len(units), "params_per_unit": units[0].P,
                           "R": R, "mode": "FSDP2 per-parameter", "storage": "bf16 params/grads, "
                           "fp32 master/m/v", "step": "per unit: all-gather+unflatten, then "
                           "reduce-scatter+AdamW", "bytes_per_step": step_bytes,
                           "l2": "inputs larger than L2 (>= 3.9 GB streamed per launch); no flush",
                           "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
                "pct_of_hbm_peak": round(value / world / peak, 4),
                "roofline": roofline, "roofline_all_gather": roofline_ag, "ddp_all_reduce": ddp,
                "grad_accumulation": accumulation, "pack": pack,
                "l2_resident_configs": small,
                "clocks": clocks.summary(), "gpu_launches": launches,
                "cpu_baseline": cpu, "e2e": e2e}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def small_configs(dev, hp):
    """The smaller workloads, whose units fit in the 129 MB L2: one 512/8/2048
    TransformerBlock (FSDP2, R=4) and twelve of them as FSDP1 FlatParameters
    (R=4). Flagged as L2-resident; they are parity workloads, reported for
    context, not the headline."""
    import torch
    from fully_sharded_state_gb300 import ShardedUnit, synth
    out = {}
    for name in ("block", "block12_flat"):
        wl = synth.WORKLOADS[name]
        units = [ShardedUnit(wl.unit_shapes(u), wl.R, wl.mode, "bf16", "bf16", device=dev)
                 for u in range(len(wl.units))]
        grads = []
        for u, U in enumerate(units):
            U.shard_from_full(synth.device_normal(synth.seed("w", wl, u), U.P, wl.w_std, dev))
            grads.append([synth.device_normal(synth.seed("g", wl, u, r), U.P, wl.g_std, dev,
                                              torch.bfloat16) for r in range(wl.R)])
        full = [torch.empty(units[0].P, dtype=torch.bfloat16, device=dev) for _ in range(wl.R)]

        def step():
            for k, U in enumerate(units):
                U.all_gather(full)
                U.reduce_scatter_adamw(grads[k], hp)

        for _ in range(5):
            step()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record()
        for _ in range(50):
            step()
        b.record()
        b.synchronize()
        ms = a.elapsed_time(b) / 50
        nbytes = sum(all_gather_bytes(U.P, wl.R) + rs_adamw_bytes(U.P, wl.R) for U in units)
        out[name] = {"units": len(units), "params_per_unit": units[0].P, "R": wl.R,
                     "mode": wl.mode, "ms_per_step": round(ms, 4),
                     "value": round(nbytes / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
                     "l2_resident": True, "gpu_launches_per_step": 2 * len(units)}
        del units, grads, full
    return out


def run_e2e(args, units, grads, full, hp, stream, dev, world, step_bytes):
    """The same step through the public API from host buffers. Every step
    copies each unit's R gradients from pinned host memory to the device on a
    copy stream (each unit's copy waits only for the previous step's
    reduce-scatter of that unit, so copies run ahead of the kernels), runs
    the unit's all-gather and reduce-scatter + AdamW once its copy is done,
    and reads its updated bf16 parameter shards back into pinned host memory
    on a third stream."""
    import torch
    R = units[0].R
    P_max = max(U.P for U in units)
    h_grads = [torch.empty(P_max, dtype=torch.bfloat16).pin_memory() for _ in range(R)]
    for r in range(R):
        h_grads[r].copy_(grads[0][r][:P_max].cpu())
    h_out = [[torch.empty(U.S, dtype=torch.bfloat16).pin_memory() for _ in range(R)]
             for U in units]
    h2d = sum(R * U.P * 2 for U in units)
    d2h = sum(R * U.S * 2 for U in units)
    steps = max(2, min(args.steps, args.e2e_steps))
    h2d_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)
    rs_done = [torch.cuda.Event() for _ in units]
    d2h_done = [torch.cuda.Event() for _ in units]
    for e in rs_done + d2h_done:
        e.record(stream)

    def e2e_step():
        copied = []
        for k, U in enumerate(units):
            h2d_stream.wait_event(rs_done[k])  # the buffer's last reader
            with torch.cuda.stream(h2d_stream):
                for r in range(R):
                    grads[k][r].copy_(h_grads[r][:U.P], non_blocking=True)
            e = torch.cuda.Event()
            e.record(h2d_stream)
            copied.append(e)
        for k, U in enumerate(units):
            stream.wait_event(copied[k])
            stream.wait_event(d2h_done[k])  # last step's read-back of this unit's shards
            U.all_gather([f[:U.P] for f in full], stream=stream)
            U.reduce_scatter_adamw(grads[k], hp, stream=stream)
            rs_done[k].record(stream)
            d2h_stream.wait_event(rs_done[k])
            with torch.cuda.stream(d2h_stream):
                for r in range(R):
                    h_out[k][r].copy_(U.param_shard[r], non_blocking=True)
            d2h_done[k].record(d2h_stream)

    e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    dt = max_over_ranks(time.perf_counter() - t0, world)
    return {"value": round(world * step_bytes * steps / dt / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(1e3 * dt / steps, 3),
            "h2d_GBps": round(h2d * steps / dt / 1e9, 1),
            "path": "pinned host grads -> device on a copy stream running ahead, per-unit "
                    "all-gather + reduce-scatter/AdamW on the compute stream, bf16 shards -> "
                    "pinned host on a third stream; host wall clock"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama4", choices=["llama4", "llama_attn"])
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-small", action="store_true", help="skip the L2-resident configs")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
