"""Each plausible mistake planted in a copy of the C oracle must fail a pin.

The copies are compiled into a temporary directory and exercised in child
processes (CPU only); the real oracle is untouched.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path


REPO = Path(__file__).resolve().parent.parent
SRC = (REPO / "oracle" / "fsdp_oracle.c").read_text()

# (name, text in the oracle, replacement)
MUTANTS = [
    ("floor instead of ceil in rank rows",
     "int64_t s = (d0 + R - 1) / R;", "int64_t s = d0 / R;"),
    ("floor instead of ceil in the layout",
     "int64_t s = (d0[i] + R - 1) / R;", "int64_t s = d0[i] / R;"),
    ("no segment padding",
     "seg = (seg + ORC_SEG_ALIGN - 1) / ORC_SEG_ALIGN * ORC_SEG_ALIGN;", "seg = seg;"),
    ("flat shard rounded down",
     "int64_t S = (total + R - 1) / R;", "int64_t S = total / R + (total % R != 0) * 0;"),
    ("gather reads the next rank's shard",
     "const char *src = (const char *)shard[r] + shard_off[i] * esize;",
     "const char *src = (const char *)shard[(r + 1) % R] + shard_off[i] * esize;"),
    ("gather ignores the segment offset",
     "const char *src = (const char *)shard[r] + shard_off[i] * esize;",
     "const char *src = (const char *)shard[r];"),
    ("pack takes rows, not elements",
     "const float *src = full + full_off[i] + start * inner[i];",
     "const float *src = full + full_off[i] + start;"),
    ("flat pack uses the wrong stride",
     "int64_t j = r * shard_numel + k;", "int64_t j = r * (shard_numel - 1) + k;"),
    ("reduction drops rank 1",
     "for (int64_t q = 1; q < R; q++)\n            acc = acc +",
     "for (int64_t q = 2; q < R; q++)\n            acc = acc +"),
    ("reduction starts from +0",
     "float acc = load_as_f32(g[0], dtype, k);\n        for (int64_t q = 1; q < R; q++)",
     "float acc = 0.0f;\n        for (int64_t q = 0; q < R; q++)"),
    ("sum without the 1/R average",
     "out[k] = acc * inv_R;", "out[k] = acc;"),
    ("average by division instead of fl(1/R)",
     "out[k] = acc * inv_R;", "out[k] = acc / (float)R;"),
    ("reduce-scatter reads the parameter start for every rank",
     "int64_t j = full_off[i] + start * inner[i];", "int64_t j = full_off[i];"),
    ("no weight decay",
     "float wk = w[k] * decay;", "float wk = w[k];"),
    ("update with the wrong sign",
     "wk = wk - step_size * (mk / denom);", "wk = wk + step_size * (mk / denom);"),
    ("no first-moment bias correction",
     "float step_size = (float)(lr / (1.0 - pow(beta1, (double)t)));",
     "float step_size = (float)lr;"),
    ("no second-moment bias correction",
     "float denom = sqrtf(vk) / bc2_sqrt + epsf;", "float denom = sqrtf(vk) + epsf;"),
    ("eps inside the square root",
     "float denom = sqrtf(vk) / bc2_sqrt + epsf;",
     "float denom = sqrtf(vk + epsf) / bc2_sqrt;"),
    ("first moment decays with beta2",
     "float mk = b1 * m[k] + one_minus_b1 * gk;", "float mk = b2 * m[k] + one_minus_b1 * gk;"),
    ("second moment of g, not g^2",
     "float vk = b2 * v[k] + one_minus_b2 * (gk * gk);",
     "float vk = b2 * v[k] + one_minus_b2 * (gk);"),
    ("bias correction one step ahead",
     "float step_size = (float)(lr / (1.0 - pow(beta1, (double)t)));",
     "float step_size = (float)(lr / (1.0 - pow(beta1, (double)(t + 1))));"),
    ("bf16 narrowing truncates",
     "u += 0x7fffu + keep_lsb;", "u += 0u * keep_lsb;"),
    ("bf16 narrowing rounds half up",
     "u += 0x7fffu + keep_lsb;", "u += 0x8000u + 0u * keep_lsb;"),
    ("owner index ignores the rank's first row",
     "index[k] = shard_off[i] + (e - full_off[i]) - start * inner[i];",
     "index[k] = shard_off[i] + (e - full_off[i]);"),
    ("flat owner uses the unpadded size",
     "rank[k] = e / S;", "rank[k] = e / (P / R > 0 ? P / R : 1); if (rank[k] >= R) rank[k] = R - 1;"),
    ("all-reduce writes only rank 0's output",
     "        for (int64_t d = 0; d < R; d++) {\n            if (out_dtype == ORC_BF16)",
     "        for (int64_t d = 0; d < 1; d++) {\n            if (out_dtype == ORC_BF16)"),
    ("all-reduce reads one element off",
     "ptrs[q] = (const char *)grad[q] + j * esize;\n        orc_sum_ranks",
     "ptrs[q] = (const char *)grad[q] + (j + 1 < P ? j + 1 : j) * esize;\n        orc_sum_ranks"),
    ("accumulation ignores the first flag",
     "            if (first)\n                acc[q][j] = g;",
     "            if (0)\n                acc[q][j] = g;"),
    ("accumulation overwrites instead of adding",
     "                acc[q][j] = acc[q][j] + g;", "                acc[q][j] = g;"),
    ("ZeRO-3 part never advances",
     "        if (filled >= target && part < R - 1) {", "        if (0) {"),
    ("ZeRO-3 segments not placed per owner",
     "            shard_off[i] = used[owner[i]];", "            shard_off[i] = used[0];"),
    ("ZeRO-3 rows held by every rank",
     "        return owner[i] == r ? d0[i] : 0;", "        return r == 0 || owner[i] == r ? d0[i] : 0;"),
    ("bf16 widening takes the low half",
     "uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h;"),
]

# A mutant may write out of bounds inside its own child process, so the child
# leaves with os._exit as soon as a pin fails, before any interpreter teardown.
_RUNNER = r"""
import os, sys
sys.path[:0] = [{repo!r}, {tests!r}]
import oracle
oracle.use_library({lib!r})
import pins
for check in pins.ALL_CHECKS:
    try:
        check()
    except Exception as exc:  # a pin that fails or errors out on the mutant
        print("caught by", check.__name__, type(exc).__name__, flush=True)
        os._exit(3)
print("not caught")
sys.exit(0)
"""


def _run_mutant(tmp: str, idx: int, old: str, new: str):
    assert SRC.count(old) == 1, f"mutant text not unique in the oracle: {old!r}"
    src = os.path.join(tmp, f"m{idx}.c")
    lib = os.path.join(tmp, f"m{idx}.so")
    Path(src).write_text(SRC.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-w",
                    "-o", lib, src, "-lm"], check=True)
    code = _RUNNER.format(repo=str(REPO), tests=str(REPO / "tests"), lib=lib)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         timeout=600)
    return res.returncode, res.stdout + res.stderr[-2000:]


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            futs = [ex.submit(_run_mutant, tmp, k, old, new)
                    for k, (_, old, new) in enumerate(MUTANTS)]
            results = [f.result() for f in futs]
    missed = [(name, out) for (name, _, _), (rc, out) in zip(MUTANTS, results) if rc != 3]
    assert not missed, "pins missed planted mistakes: " + "; ".join(n for n, _ in missed)
