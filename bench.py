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
                    [--no-configs] [--no-memory] [--no-ceilings]
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


def rs_kernel_name(shapes, R: int, grad_b: int, sms: int) -> str:
    """The reduce-scatter + AdamW kernel the library launches for one FSDP2
    unit: the staged one (gradient slices by cp.async.bulk) when the R
    gradient streams carry at least 8 bytes per element, a stage (R slices of
    a 2,048-element tile) fits in 32 KB and the launch has at least 32 tiles
    per staged thread block (2 per SM), or 16 when at most half of its
    elements sit in rank pieces that start on the 8-element grid; the
    register one otherwise."""
    tiles = elems = aligned8 = 0
    full_off = 0
    for s in shapes:
        inner = 1
        for x in s[1:]:
            inner *= x
        rows = -(-s[0] // R)
        for r in range(R):
            n = max(0, min(rows, s[0] - r * rows)) * inner
            tiles += -(-n // 2048)
            elems += n
            if (full_off + r * rows * inner) % 8 == 0:  # shard offsets are always
                aligned8 += n
        full_off += s[0] * inner
    per_cta = 16 if 2 * aligned8 < elems else 32
    if (R in (2, 4, 8) and R * grad_b >= 8 and R * 2048 * grad_b <= 32 * 1024
            and tiles >= per_cta * 2 * sms):
        return "rs_adamw_staged_kernel"
    return "rs_adamw_kernel"


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


def cpu_baseline(wl, shapes, w_dev, grads_dev):
    """The CPU oracle timed on one whole unit of the GPU arm's own inputs (its
    device-generated weights and R gradients, copied to the host): once with
    the plain single-thread build, then with the OpenMP build of the same
    source on all host cores, whose outputs must be bit-identical."""
    import oracle
    R = wl.R
    O = oracle.layout(oracle.PER_PARAM, R, shapes)
    P, S = O.full_numel, O.shard_numel
    w = w_dev.detach().cpu().numpy()
    grads = [g.detach().view(torch_int16()).cpu().numpy().view(np.uint16) for g in grads_dev]
    hp = oracle.AdamWHP(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay)
    masters0, p16_0 = oracle.pack(O, w, with_bf16=True)
    del w
    nbytes = all_gather_bytes(P, R) + rs_adamw_bytes(P, R)

    def one_run():
        masters = [x.copy() for x in masters0]
        m = [np.zeros(S, np.float32) for _ in range(R)]
        v = [np.zeros(S, np.float32) for _ in range(R)]
        t0 = time.perf_counter()
        full = oracle.all_gather(O, p16_0)
        _, p16 = oracle.rs_adamw(O, grads, masters, m, v, hp, 1, with_bf16=True)
        dt = time.perf_counter() - t0
        return dt, full, masters, m, v, p16

    dt1, *single = one_run()
    with oracle.using(oracle.build(openmp=True)):
        runs = [one_run() for _ in range(3)]
    dt_omp = statistics.median(r[0] for r in runs)
    omp = runs[-1][1:]
    identical = all(np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))
                    for xs, ys in zip(single, omp) for a, b in zip(xs, ys))
    cores = os.cpu_count()
    desc = (f"one whole unit of the benchmark ({P:,} params, R={R}) on the GPU arm's own "
            "inputs: oracle all-gather + reduce-scatter/AdamW")
    return {"value": round(nbytes / dt1 / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": desc + ", single thread", "seconds": round(dt1, 3),
            "openmp": {"value": round(nbytes / dt_omp / 1e9, 4), "unit": UNIT, "cores": cores,
                       "seconds_median_of_3": round(dt_omp, 3),
                       "bit_identical_to_single_thread": bool(identical),
                       "build": "same oracle source, gcc -fopenmp (element loops split over "
                                "threads)"},
            "host_cores_available": cores, "host_cpu": host_cpu()}


def torch_int16():
    import torch
    return torch.int16


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

NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


def roofline_entry(kernel, nbytes, ms, peak, peak_src, traffic=None, ceilings=None):
    """Roofline record of one kernel: algorithmic bytes per launch over its
    mean CUDA-event launch time, as a fraction of the measured HBM copy peak,
    of the nominal HBM bandwidth and (when measured in the run) of the
    write-only stream ceiling."""
    gbs = nbytes / (ms * 1e-3) / 1e9
    e = {"kernel": kernel, "bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
         "unit": "GB/s", "frac": round(gbs / peak, 4), "peak_source": peak_src,
         "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
         "nominal_peak": NOMINAL_HBM_GBS, "algorithmic_bytes_per_launch": int(nbytes),
         "avg_launch_ms": round(ms, 4), "traffic": traffic}
    if ceilings and ceilings.get("write_only_x_R_gbs"):
        e["frac_of_write_ceiling"] = round(gbs / ceilings["write_only_x_R_gbs"], 4)
    return e


def timed_back_to_back(torch, stream, fn, n=50, warm=5):
    """CUDA-event time (ms) per call of fn() issued n times back to back on
    `stream` (throughput: the host issues ahead while the GPU works)."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        fn()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / n


def timed_launches(torch, stream, fn, n=20, warm=3):
    """Mean CUDA-event time (ms) of fn() on `stream`, each launch bracketed."""
    for _ in range(warm):
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


def measure_ceilings(torch, dev, stream, full, grads0, h_grads):
    """Stream ceilings measured in the same run, for reading the kernels'
    fractions: a write-only stream over R full-unit bf16 buffers with the
    all-gather's store pattern (the library's fsdp_write_stream helper; the
    write side that bounds the gather and the all-reduce), torch's own fill
    kernels on the same buffers for comparison, a device copy of R buffers,
    and the pinned host <-> device link (copy engines) on every unit's R
    host gradient buffers."""
    from fully_sharded_state_gb300 import capi
    R = len(full)
    P = full[0].numel()
    with torch.cuda.stream(stream):
        wr = timed_launches(torch, stream, lambda: capi.fsdp_write_stream(full, stream=stream),
                            n=10)
        zero = timed_launches(torch, stream, lambda: [f.zero_() for f in full], n=10)
        fill = timed_launches(torch, stream, lambda: [f.fill_(1.5) for f in full], n=10)
        cp = timed_launches(torch, stream,
                            lambda: [f.copy_(g[:P]) for f, g in zip(full, grads0)], n=10)
        h2d = [timed_launches(torch, stream,
                              lambda hu=hu: [f[:h.numel()].copy_(h, non_blocking=True)
                                             for f, h in zip(full, hu)], n=3, warm=1)
               for hu in h_grads]
        d2h = timed_launches(torch, stream, lambda: [h.copy_(f[:h.numel()], non_blocking=True)
                                                     for f, h in zip(full, h_grads[0])], n=3)
    nh = [sum(h.numel() * 2 for h in hu) for hu in h_grads]
    gbs = lambda b, ms: round(b / (ms * 1e-3) / 1e9, 1)
    return {"write_only_x_R_gbs": gbs(R * P * 2, wr),
            "torch_zero_x_R_gbs": gbs(R * P * 2, zero), "torch_fill_x_R_gbs": gbs(R * P * 2, fill),
            "device_copy_x_R_gbs": gbs(R * P * 4, cp),
            "h2d_pinned_gbs": gbs(nh[0], h2d[0]),
            "h2d_pinned_gbs_per_unit": [gbs(b, ms) for b, ms in zip(nh, h2d)],
            "d2h_pinned_gbs": gbs(nh[0], d2h),
            "how": f"fsdp_write_stream (32-byte stores, the gather's grid) and torch zero_ / "
                   f"fill_ over {R} x {P:,} bf16; torch copy_ of {R} x {P:,} bf16 "
                   f"(read + write bytes); pinned host <-> device copies of each unit's {R} x "
                   f"{P:,} bf16 gradients; CUDA events, mean of 10 (3 for host copies)"}


def peak_memory(torch, dev, unit_shapes, R, mode, hp, seed=11):
    """Peak device memory of one training step of the engine against the
    FSDP2 page's formula (§01): M_peak ~= M_shard + M_largest_unsharded +
    M_prefetch + M_a + M_temp. Per unit and for all R virtual ranks (they
    share this GPU): M_shard = R*S*14 B (bf16 shard, fp32 master, m, v; the
    reduce-scatter's fp32 output lives in registers, so no sharded gradient
    is stored); the largest unsharded unit = R full bf16 buffers; the
    prefetch buffer = one more set (prefetch schedule only); M_temp = one
    unit's R full bf16 gradients, which exist from the unit's backward to its
    reduce-scatter; no activations. Two schedules of one step: forward
    gathers every unit, backward walks the units in reverse, re-gathers each
    one, produces its gradients and reduce-scatters them; "prefetch" issues
    the next unit's gather together with the current unit's reduce-scatter
    (fsdp_reduce_scatter_adamw_gather) into a second set of full buffers.
    measured = peak of the bytes requested from torch's allocator during the
    step; allocator_bytes = its max_memory_allocated (with block rounding)."""
    from fully_sharded_state_gb300 import ShardedUnit

    def requested(key):
        # bytes the program asked for (the allocator's own rounding and
        # segment slack are left out; max_memory_allocated counts them)
        return torch.cuda.memory_stats(dev).get(f"requested_bytes.all.{key}", 0)

    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    base = requested("current")
    base_alloc = torch.cuda.memory_allocated(dev)
    units = []
    for u, shapes in enumerate(unit_shapes):
        U = ShardedUnit(shapes, R, mode, "bf16", "bf16", device=dev)
        w = torch.empty(U.P, dtype=torch.float32, device=dev).normal_(0.0, 0.02)
        U.shard_from_full(w)
        del w
        units.append(U)
    torch.cuda.synchronize(dev)
    P_max = max(U.P for U in units)
    m_shard = sum(R * U.S * (2 + 4 + 4 + 4) for U in units)
    out = {}
    for schedule in ("in_order", "prefetch"):
        torch.cuda.synchronize(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        nsets = 2 if schedule == "prefetch" else 1
        sets = [[torch.empty(P_max, dtype=torch.bfloat16, device=dev) for _ in range(R)]
                for _ in range(nsets)]
        view = lambda k, U: [f[:U.P] for f in sets[k % nsets]]
        for k, U in enumerate(units):  # forward
            U.all_gather(view(k, U))
        n = len(units)
        if schedule == "in_order":
            for k in reversed(range(n)):  # backward
                U = units[k]
                U.all_gather(view(k, U))
                g = [torch.empty(U.P, dtype=torch.bfloat16, device=dev).normal_(0.0, 1e-3)
                     for _ in range(R)]
                U.reduce_scatter_adamw(g, hp)
                del g
        else:
            units[n - 1].all_gather(view(n - 1, units[n - 1]))
            for k in reversed(range(n)):
                U = units[k]
                g = [torch.empty(U.P, dtype=torch.bfloat16, device=dev).normal_(0.0, 1e-3)
                     for _ in range(R)]
                if k > 0:
                    U.reduce_scatter_adamw_and_gather(g, hp, units[k - 1],
                                                      view(k - 1, units[k - 1]))
                else:
                    U.reduce_scatter_adamw(g, hp)
                del g
        torch.cuda.synchronize(dev)
        measured = requested("peak") - base
        allocated = torch.cuda.max_memory_allocated(dev) - base_alloc
        largest = R * P_max * 2
        formula = m_shard + largest + (largest if nsets == 2 else 0) + R * P_max * 2
        out[schedule] = {"measured_bytes": int(measured), "formula_bytes": int(formula),
                         "allocator_bytes": int(allocated),
                         "M_shard": int(m_shard), "M_largest_unsharded": int(largest),
                         "M_prefetch": int(largest if nsets == 2 else 0),
                         "M_temp_gradients": int(R * P_max * 2), "M_activations": 0,
                         "measured_over_formula": round(measured / formula, 6)}
        del sets
    del units
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return out


def config_entry(torch, dev, stream, name, hp, peak, peak_src):
    """One workload of the benchmark's configurations, timed as a training
    step (every unit's all-gather + unflatten, then its reduce-scatter +
    AdamW) with plain per-unit calls and, for several units, with the
    prepared multi-unit calls (two launches per step); 50 steps back to back
    between two CUDA events."""
    from fully_sharded_state_gb300 import (ShardedUnit, prepare_all_gather_units,
                                           prepare_reduce_scatter_adamw_units, synth)
    wl = synth.WORKLOADS[name]
    R = wl.R
    bf16p, bf16g = wl.param_dtype == "bf16", wl.grad_dtype == "bf16"
    pb, gb = (2 if bf16p else 4), (2 if bf16g else 4)
    units, grads = [], []
    for u in range(len(wl.units)):
        U = ShardedUnit(wl.unit_shapes(u), R, wl.mode, wl.param_dtype, wl.grad_dtype, device=dev)
        U.shard_from_full(synth.device_weights(wl, u, dev))
        units.append(U)
        grads.append(synth.device_grads(wl, u, dev))
    fulls = [U.alloc_full() for U in units]
    ag = sum(all_gather_bytes(U.P, R, pb) for U in units)
    rs = sum(rs_adamw_bytes(U.P, R, gb, 2 if bf16p else 0) for U in units)
    distinct = sum(R * U.P * (gb + pb) + R * U.S * (12 + (2 if bf16p else 0)) for U in units)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def step():
        for k, U in enumerate(units):
            U.all_gather(fulls[k], stream=stream)
            U.reduce_scatter_adamw(grads[k], hp, stream=stream)

    ms = timed_back_to_back(torch, stream, step)
    gbs = (ag + rs) / (ms * 1e-3) / 1e9
    # each kernel on its own, every unit once per pass
    ms_ag = timed_back_to_back(torch, stream, lambda: [U.all_gather(fulls[k], stream=stream)
                                                       for k, U in enumerate(units)])
    ms_rs = timed_back_to_back(torch, stream, lambda: [U.reduce_scatter_adamw(grads[k], hp,
                                                                              stream=stream)
                                                       for k, U in enumerate(units)])
    kernels = {name: {"ms": round(t, 4), "algorithmic_bytes": int(nb),
                      "achieved": round(nb / (t * 1e-3) / 1e9, 1),
                      "frac": round(nb / (t * 1e-3) / 1e9 / peak, 4)}
               for name, t, nb in (("all_gather", ms_ag, ag), ("rs_adamw", ms_rs, rs))}
    e = {"workload": name, "cfg": wl.cfg, "units": len(units), "params_per_unit": units[0].P,
         "R": R, "mode": wl.mode, "dtypes": f"{wl.param_dtype} params / {wl.grad_dtype} grads",
         "algorithmic_bytes_per_step": int(ag + rs), "distinct_bytes": int(distinct),
         "l2_resident": bool(distinct < l2), "ms_per_step": round(ms, 4),
         "achieved": round(gbs, 1), "unit": UNIT, "frac": round(gbs / peak, 4),
         "peak_source": peak_src, "gpu_launches_per_step": 2 * len(units),
         "calls": "plain per-unit calls", "per_kernel": kernels}
    if len(units) == 1:
        U, g, f = units[0], grads[0], fulls[0]
        ag1, rs1 = U.prepare_all_gather(f), U.prepare_reduce_scatter_adamw(g)
        ms_p = timed_back_to_back(torch, stream, lambda: (ag1(stream=stream),
                                                          rs1(hp, stream=stream)))
        gbs_p = (ag + rs) / (ms_p * 1e-3) / 1e9
        e["prepared_calls"] = {"ms_per_step": round(ms_p, 4), "achieved": round(gbs_p, 1),
                               "frac": round(gbs_p / peak, 4), "gpu_launches_per_step": 2,
                               "calls": "prepared per-unit calls"}
        del ag1, rs1
    if len(units) > 1:
        ag_call = prepare_all_gather_units(units, fulls)
        rs_call = prepare_reduce_scatter_adamw_units(units, grads)

        def step_units():
            ag_call(stream=stream)
            rs_call(hp, stream=stream)

        ms_u = timed_back_to_back(torch, stream, step_units)
        gbs_u = (ag + rs) / (ms_u * 1e-3) / 1e9
        e["all_units_per_call"] = {"ms_per_step": round(ms_u, 4), "achieved": round(gbs_u, 1),
                                   "frac": round(gbs_u / peak, 4), "gpu_launches_per_step": 2,
                                   "calls": "prepared multi-unit calls"}
    if not e["l2_resident"] and ms > 0 and gbs < 0.5 * peak:
        e["note"] = "launch-latency bound (small units)"
    if name == "toy":
        e["note"] = "eight elements per step: launch-latency bound, reported for completeness"
    del units, grads, fulls
    return e


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
    stream = torch.cuda.current_stream(dev)
    peak, peak_src = measured_peak()

    memory = None
    if not args.no_memory:
        memory = peak_memory(torch, dev, [[s for _, s in spec] for spec in units_spec], R,
                             "per_param", hp)

    units, grads, pack_ms = [], [], []
    w_unit0 = None
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
        if u == 0 and rank == 0 and world == 1 and not args.no_cpu_baseline:
            w_unit0 = w_full.cpu()
        del w_full
        units.append(U)
        grads.append([synth.device_normal(synth.seed("g", wl, u, r), U.P, wl.g_std, dev,
                                          torch.bfloat16) for r in range(R)])
    P_max = max(U.P for U in units)
    full = [torch.empty(P_max, dtype=torch.bfloat16, device=dev) for _ in range(R)]

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

    ms_step = elapsed_ms / args.steps
    value = world * step_bytes / (ms_step * 1e-3) / 1e9

    # host gradients of every unit, pinned (the end-to-end leg's inputs)
    h_grads = None
    if not args.no_e2e or not args.no_ceilings:
        h_grads = [[torch.empty(U.P, dtype=torch.bfloat16).pin_memory() for _ in range(R)]
                   for U in units]
        for k, U in enumerate(units):
            for r in range(R):
                h_grads[k][r].copy_(grads[k][r])
    ceilings = None
    if not args.no_ceilings:
        ceilings = measure_ceilings(torch, dev, stream, full, grads[0], h_grads)

    def entry(kernel, nbytes, ms, traffic_key):
        return roofline_entry(kernel, nbytes, ms, peak, peak_src,
                              profiled_traffic(traffic_key, args.workload) if traffic_key
                              else None, ceilings)

    rs_name = rs_kernel_name(units[0].shapes, R, 2,
                             torch.cuda.get_device_properties(dev).multi_processor_count)
    roofline = entry(f"{rs_name} (fused reduce-scatter + AdamW)", rs_bytes / len(units),
                     statistics.mean(rs_ms), "rs_adamw")
    roofline_ag = entry("all_gather_kernel (all-gather + unflatten)", ag_bytes / len(units),
                        statistics.mean(ag_ms), "all_gather")

    # DDP's collective on the same unit, for comparison: all-reduce of the R
    # bf16 gradients into R fp32 full outputs (reduce dtype fp32)
    U0 = units[0]
    ar_out = [torch.empty(U0.P, dtype=torch.float32, device=dev) for _ in range(R)]
    ar_ms = timed_launches(torch, stream,
                           lambda: U0.all_reduce(grads[0], ar_out, "f32", stream=stream))
    ddp = entry("all_reduce_kernel (DDP all-reduce: bf16 grads -> fp32 outputs)",
                R * U0.P * (2 + 4), ar_ms, "all_reduce")
    # ZeRO-1's step on the same unit: the all-reduce above, each rank's AdamW
    # from its own averaged fp32 gradient, then the all-gather
    z1_ms = timed_launches(torch, stream,
                           lambda: U0.adamw_from_reduced(ar_out, hp, stream=stream))
    del ar_out
    z1_adamw = entry("adamw_reduced_kernel (ZeRO-1: AdamW on each rank's partition from the "
                     "all-reduced gradient)", U0.P * (4 + 24 + 2), z1_ms, None)
    zero1 = {"adamw_from_reduced": z1_adamw,
             "step_ms_per_unit": round(ar_ms + z1_ms + statistics.mean(ag_ms), 4),
             "fsdp_step_ms_per_unit": round(statistics.mean(rs_ms) + statistics.mean(ag_ms), 4),
             "algorithmic_bytes_per_param": {"zero1": 48 + 30 + 18, "fsdp": 42 + 18},
             "note": "all-reduce + AdamW from the averaged gradient + all-gather, against "
                     "the fused reduce-scatter + AdamW + all-gather; same results bit for bit"}

    # gradient accumulation on the same unit: one more micro-batch added into
    # the fp32 accumulators, and the last micro-batch fused into the step
    acc = U0.alloc_accumulators()
    U0.accumulate_grad(grads[0], acc, first=True, stream=stream)
    acc_ms = timed_launches(torch, stream,
                            lambda: U0.accumulate_grad(grads[0], acc, first=False, stream=stream))
    rsacc_ms = timed_launches(torch, stream,
                              lambda: U0.reduce_scatter_adamw_accum(acc, grads[0], hp,
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

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, units, grads, h_grads, full, hp, stream, dev, world, step_bytes)

    configs = None
    if not args.no_configs:
        configs = {"llama4": {
            "workload": "llama4", "cfg": 5, "units": len(units), "params_per_unit": U0.P,
            "R": R, "mode": "per_param", "dtypes": "bf16 params / bf16 grads",
            "algorithmic_bytes_per_step": int(step_bytes), "l2_resident": False,
            "ms_per_step": round(ms_step, 4), "achieved": round(value / world, 1), "unit": UNIT,
            "frac": round(value / world / peak, 4), "peak_source": peak_src,
            "gpu_launches_per_step": 2 * len(units), "calls": "plain per-unit calls",
            "note": "the headline workload: see value and roofline"}} \
            if args.workload == "llama4" else {}
        if configs:
            # the same four units through the prepared multi-unit calls
            from fully_sharded_state_gb300 import (prepare_all_gather_units,
                                                   prepare_reduce_scatter_adamw_units)
            fulls_u = [[f[:U.P] for f in full] if k == 0 else
                       [torch.empty(U.P, dtype=torch.bfloat16, device=dev) for _ in range(R)]
                       for k, U in enumerate(units)]
            ag_call = prepare_all_gather_units(units, fulls_u)
            rs_call = prepare_reduce_scatter_adamw_units(units, grads)
            ms_u = timed_back_to_back(torch, stream, lambda: (ag_call(stream=stream),
                                                              rs_call(hp, stream=stream)), n=20)
            gbs_u = step_bytes / (ms_u * 1e-3) / 1e9
            configs["llama4"]["all_units_per_call"] = {
                "ms_per_step": round(ms_u, 4), "achieved": round(gbs_u, 1),
                "frac": round(gbs_u / peak, 4), "gpu_launches_per_step": 2,
                "calls": "prepared multi-unit calls (all four gathers, then all four "
                         "reduce-scatters)"}
            del ag_call, rs_call, fulls_u
        for name in ("toy", "block", "block12_flat", "ragged"):
            configs[name] = config_entry(torch, dev, stream, name, hp, peak, peak_src)

    cpu = None
    if w_unit0 is not None:
        cpu = cpu_baseline(wl, [s for _, s in units_spec[0]], w_unit0, grads[0])

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
                "pct_of_nominal_hbm": round(value / world / NOMINAL_HBM_GBS, 4),
                "roofline": roofline, "roofline_all_gather": roofline_ag, "ddp_all_reduce": ddp,
                "zero1": zero1,
                "grad_accumulation": accumulation, "pack": pack, "ceilings": ceilings,
                "configs": configs, "peak_memory": memory,
                "clocks": clocks.summary(), "gpu_launches": launches,
                "cpu_baseline": cpu, "e2e": e2e}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, units, grads, h_grads, full, hp, stream, dev, world, step_bytes):
    """The same step through the public API from host buffers. Every step
    copies each unit's own R gradients from pinned host memory to the device
    on two copy streams (each unit's copy waits only for the previous step's
    reduce-scatter of that unit, so copies run ahead of the kernels), runs
    the unit's all-gather and reduce-scatter + AdamW once its copy is done,
    and reads its updated bf16 parameter shards back into pinned host memory
    on a third stream. As many steps as the device-timed region."""
    import torch
    R = units[0].R
    h_out = [[torch.empty(U.S, dtype=torch.bfloat16).pin_memory() for _ in range(R)]
             for U in units]
    h2d = sum(R * U.P * 2 for U in units)
    d2h = sum(R * U.S * 2 for U in units)
    steps = args.steps
    # two copy streams: one stream's host-to-device copies reach ~178 GB/s on
    # GB300, two together the link's ~211 GB/s
    h2d_streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    d2h_stream = torch.cuda.Stream(dev)
    rs_done = [torch.cuda.Event() for _ in units]
    d2h_done = [torch.cuda.Event() for _ in units]
    for e in rs_done + d2h_done:
        e.record(stream)

    def e2e_step():
        copied = []
        for k, U in enumerate(units):
            evs = []
            for c, hs in enumerate(h2d_streams):
                hs.wait_event(rs_done[k])  # the buffer's last reader
                with torch.cuda.stream(hs):
                    for r in range(c, R, len(h2d_streams)):
                        grads[k][r].copy_(h_grads[k][r], non_blocking=True)
                e = torch.cuda.Event()
                e.record(hs)
                evs.append(e)
            copied.append(evs)
        for k, U in enumerate(units):
            for e in copied[k]:
                stream.wait_event(e)
            stream.wait_event(d2h_done[k])  # last step's read-back of this unit's shards
            U.all_gather([f[:U.P] for f in full], stream=stream)
            U.reduce_scatter_adamw(grads[k], hp, stream=stream)
            rs_done[k].record(stream)
            d2h_stream.wait_event(rs_done[k])
            with torch.cuda.stream(d2h_stream):
                for r in range(R):
                    h_out[k][r].copy_(U.param_shard[r], non_blocking=True)
            d2h_done[k].record(d2h_stream)

    def link_gbs():
        # the host link over the same buffers, with no kernels: every unit's
        # gradients copied once on the two copy streams
        torch.cuda.synchronize(dev)
        t = time.perf_counter()
        for k in range(len(units)):
            for c, hs in enumerate(h2d_streams):
                with torch.cuda.stream(hs):
                    for r in range(c, R, len(h2d_streams)):
                        grads[k][r].copy_(h_grads[k][r], non_blocking=True)
        torch.cuda.synchronize(dev)
        return round(h2d / (time.perf_counter() - t) / 1e9, 1)

    e2e_step()
    link_before = link_gbs()
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    dt = max_over_ranks(time.perf_counter() - t0, world)
    link_after = link_gbs()
    return {"value": round(world * step_bytes * steps / dt / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(1e3 * dt / steps, 3),
            "h2d_GBps": round(h2d * steps / dt / 1e9, 1),
            "h2d_link_GBps_before_after": [link_before, link_after],
            "path": "each unit's own pinned host grads -> device on two copy streams running "
                    "ahead, per-unit all-gather + reduce-scatter/AdamW on the compute stream, "
                    "bf16 shards -> pinned host on a fourth stream; host wall clock"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama4", choices=["llama4", "llama_attn"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-memory", action="store_true", help="skip the peak-memory step")
    ap.add_argument("--no-ceilings", action="store_true", help="skip the stream ceilings")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
