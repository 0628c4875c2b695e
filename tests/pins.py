"""Pins of the CPU oracle to what the pages and the mathematics fix.

Each ``check_*`` function raises AssertionError when the oracle disagrees with
a printed value (fixtures under ``tests/golden/``, each citing its page), a
closed form, an invariant, a library routine on a special case, or a brute
force over tiny inputs. ``test_oracle_pins.py`` runs them against the oracle;
``test_oracle_mutants.py`` runs them against copies of the oracle with a
planted mistake and requires that some check fails for each.
"""
from __future__ import annotations

from fractions import Fraction
from pathlib import Path

import numpy as np

import oracle
from oracle import brute, formulas

GOLDEN = Path(__file__).parent / "golden"
HP = oracle.AdamWHP(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def golden(name: str) -> dict:
    out = {}
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.split("#", 1)[0].strip()
        if line:
            key, val = line.split(":", 1)
            out[key.strip()] = val.strip()
    return out


def ints(text: str) -> list:
    return [int(x) for x in text.split()]


def _owned(L, r, i, buf):
    """Rank r's real elements of parameter i inside its shard buffer."""
    _, rows = L.rank_rows(i, r)
    o = int(L.shard_off[i])
    return buf[o:o + rows * int(L.inner[i])]


def _tiny_shapes(rng, max_params=4):
    shapes = []
    for _ in range(int(rng.integers(1, max_params + 1))):
        ndim = int(rng.integers(1, 4))
        shp = [int(rng.integers(0, 10))] + [int(rng.integers(1, 5)) for _ in range(ndim - 1)]
        shapes.append(tuple(shp))
    return shapes


# ---------------------------------------------------------------------------
# "FSDP Training Step Walkthrough"
# ---------------------------------------------------------------------------

def check_walkthrough_layout_and_gather():
    g = golden("walkthrough_toy.txt")
    R = int(g["R"])
    for unit in ("W1", "W2"):
        full = np.array(ints(g[f"unit {unit}"]), np.float32)
        L = oracle.layout(oracle.PER_PARAM, R, [full.shape])
        masters, _ = oracle.pack(L, full, with_bf16=False)
        for r in range(R):
            assert _owned(L, r, 0, masters[r]).tolist() == ints(g[f"shard rank{r} {unit}"])
            own = _owned(L, r, 0, masters[r]).size
            assert not masters[r][own:].any(), "padding must be zero"
        for d, out in enumerate(oracle.all_gather(L, masters)):
            assert out.tolist() == ints(g[f"gather {unit}"]), d


def check_walkthrough_reduce_scatter():
    g = golden("walkthrough_toy.txt")
    R = int(g["R"])
    names = ints(g["unit W2"])
    # rank q's gradient of w_k: (q + 1) * k + q / 4 (distinct, exact in fp32)
    grads = [np.array([(q + 1) * k + 0.25 * q for k in names], np.float32) for q in range(R)]
    L = oracle.layout(oracle.PER_PARAM, R, [(len(names),)])
    gsh = oracle.reduce_scatter(L, grads)
    for r in range(R):
        ks = ints(g[f"rs-avg rank{r} W2"])
        expect = [Fraction(sum(Fraction(q + 1) * k + Fraction(q, 4) for q in range(R)), R)
                  for k in ks]
        assert [Fraction(float(x)) for x in _owned(L, r, 0, gsh[r])] == expect


def check_walkthrough_step_matches_single_device_adamw():
    """Sharded step == one AdamW step of torch on the full unit with the rank
    average of the gradients; each rank updates exactly the parameters its row
    of the optimizer table names."""
    import torch
    g = golden("walkthrough_toy.txt")
    R = int(g["R"])
    rng = np.random.default_rng(7)
    names = {"W1": ints(g["unit W1"]), "W2": ints(g["unit W2"])}
    updated = {}
    for unit, ks in names.items():
        w0 = rng.standard_normal(len(ks)).astype(np.float32)
        grads = [rng.standard_normal(len(ks)).astype(np.float32) for _ in range(R)]
        L = oracle.layout(oracle.PER_PARAM, R, [w0.shape])
        master, _ = oracle.pack(L, w0, with_bf16=False)
        m = [np.zeros(L.shard_numel, np.float32) for _ in range(R)]
        v = [np.zeros(L.shard_numel, np.float32) for _ in range(R)]
        oracle.rs_adamw(L, grads, master, m, v, HP, 1, with_bf16=False)
        full_after = oracle.all_gather(L, master)[0]

        p = torch.nn.Parameter(torch.from_numpy(w0.copy()))
        p.grad = torch.from_numpy(np.mean(np.stack(grads).astype(np.float64), 0).astype(np.float32))
        opt = torch.optim.AdamW([p], lr=HP.lr, betas=(HP.beta1, HP.beta2), eps=HP.eps,
                                weight_decay=HP.weight_decay, foreach=False)
        opt.step()
        ref = p.detach().numpy()
        assert np.all(np.abs(full_after - ref) <= 1e-5 * np.maximum(1, np.abs(ref)))
        for r in range(R):
            own = _owned(L, r, 0, master[r])
            start, rows = L.rank_rows(0, r)
            updated.setdefault(r, []).extend(ks[start:start + rows])
            assert np.array_equal(own, full_after[start:start + rows])
    for r in range(R):
        assert updated[r] == ints(g[f"update rank{r}"])


def check_walkthrough_comm_tally():
    g = golden("walkthrough_toy.txt")
    R = int(g["R"])
    tally = formulas.fsdp_step_tally([4, 4], R)
    ops = [(ph, op, k) for ph, op, k, _ in tally]
    assert ops == [("forward", "all-gather", 0), ("forward", "all-gather", 1),
                   ("backward", "all-gather", 1), ("backward", "reduce-scatter", 1),
                   ("backward", "all-gather", 0), ("backward", "reduce-scatter", 0),
                   ("optimizer", "none", -1)]
    assert [int(x) for *_, x in tally] == ints(g["tally"])
    assert sum(x for *_, x in tally) == int(g["tally total"])
    assert formulas.allreduce_volume_per_rank(8, R) == int(g["ddp allreduce total"])


# ---------------------------------------------------------------------------
# "FSDP2 的参数全聚合、梯度归约分片与显存峰值"
# ---------------------------------------------------------------------------

def check_fsdp2_eight_params():
    g = golden("fsdp2_eight_params.txt")
    R = int(g["R"])
    w = np.array(ints(g["unit w"]), np.float32)
    L = oracle.layout(oracle.PER_PARAM, R, [w.shape])
    masters, _ = oracle.pack(L, w, with_bf16=False)
    for r in range(R):
        assert _owned(L, r, 0, masters[r]).tolist() == ints(g[f"shard rank{r} w"])
    assert all(x.tolist() == ints(g["gather w"]) for x in oracle.all_gather(L, masters))
    rng = np.random.default_rng(3)
    grads = [rng.integers(-50, 50, w.size).astype(np.float32) for _ in range(R)]
    gsh = oracle.reduce_scatter(L, grads)
    for r in range(R):
        a, b = ints(g[f"rs rank{r} range"])
        exact = [Fraction(int(sum(gq[j] for gq in grads)), R) for j in range(a, b)]
        assert [Fraction(float(x)) for x in _owned(L, r, 0, gsh[r])] == exact


def check_exercise_sum_reduce_scatter():
    """Exercise 2 of §16: SUM reduce-scatter of g0=[1,2,3,4], g1=[5,6,7,8]
    leaves [6,8] on rank 0 and [10,12] on rank 1; the global average halves
    them. The expected sums come from the brute force (exact integers)."""
    g = golden("fsdp2_eight_params.txt")
    g0, g1 = ints(g["exercise g0"]), ints(g["exercise g1"])
    R = 2
    sums = brute.reduce_scatter_sum([g0, g1], R, brute.per_param_owner_ranges([(4,)], R))
    assert sums == [[6, 8], [10, 12]]
    L = oracle.layout(oracle.PER_PARAM, R, [(4,)])
    gsh = oracle.reduce_scatter(L, [np.array(g0, np.float32), np.array(g1, np.float32)])
    for r in range(R):
        assert [Fraction(float(x)) for x in _owned(L, r, 0, gsh[r])] == \
            [Fraction(s, R) for s in sums[r]]


def check_memory_formulas():
    g = golden("memory_formulas.txt")
    W, G, O = (Fraction(g[k]) for k in ("exercise weights GB", "exercise grads GB",
                                          "exercise optimizer GB"))
    R = int(g["exercise R"])
    # with P = 1 "GB-parameter", b_w, b_g, b_o are the GB totals themselves
    steady = formulas.shard_state_bytes(1, W, G, O, R)
    assert steady == 12
    peak = formulas.peak_bytes(steady, Fraction(g["exercise largest group GB"]),
                               Fraction(g["exercise prefetch GB"]))
    assert peak == 18
    assert formulas.ddp_bytes_per_param_adamw_mixed() == int(g["ddp bytes per param"])
    assert formulas.zero3_bytes_per_param(8) == 2


# ---------------------------------------------------------------------------
# "FSDP Transformer Block Sharding Example"
# ---------------------------------------------------------------------------

def _matrices_only():
    return [(n, s) for n, s in formulas.block_shapes(with_norms=False)]


def check_block_fsdp2_table():
    g = golden("block_sharding.txt")
    R = int(g["R"])
    named = _matrices_only()
    L = oracle.layout(oracle.PER_PARAM, R, [s for _, s in named])
    for i, (name, shape) in enumerate(named):
        full_txt, per_txt, cnt_txt = (x.strip() for x in g[f"fsdp2 {name}"].split("|"))
        assert list(shape) == ints(full_txt)
        for r in range(R):
            _, rows = L.rank_rows(i, r)
            assert [rows] + list(shape[1:]) == ints(per_txt)
            assert rows * int(L.inner[i]) == int(cnt_txt)
    for r in range(R):
        assert L.rank_numel(r) == int(g["fsdp2 total per GPU"])
    assert round(L.rank_numel(0) * 2 / 1e6, 2) == float(g["fsdp2 per GPU fp16 MB approx"])
    for r in range(R):
        start, rows = L.rank_rows(0, r)
        assert [start, start + rows - 1] == ints(g[f"W_Q rows gpu{r}"])


def check_block_fsdp1_flat():
    g = golden("block_sharding.txt")
    R = int(g["R"])
    L = oracle.layout(oracle.FLAT, R, [s for _, s in _matrices_only()])
    assert L.full_numel == int(g["fsdp1 flat length"])
    assert L.shard_numel == int(g["fsdp1 flat_param size"])
    for r in range(R):
        a, b = ints(g[f"fsdp1 gpu{r}"])
        assert (r * L.shard_numel, r * L.shard_numel + L.rank_numel(r)) == (a, b)


def check_block_counts():
    g = golden("block_sharding.txt")
    shapes = dict(formulas.block_shapes(with_norms=False))
    assert formulas.numel(shapes["W_Q"]) == int(g["count W_Q"])
    assert formulas.numel(shapes["W_up"]) == int(g["count W_up"])
    assert formulas.numel(shapes["W_down"]) == int(g["count W_down"])
    block = sum(formulas.numel(s) for s in shapes.values())
    assert round(block / 1e6, 2) == float(g["block params approx M"])
    assert round(block * 2 / 1e6, 1) == float(g["block fp16 MB approx"])
    with_norms = sum(formulas.numel(s) for _, s in formulas.block_shapes(with_norms=True))
    assert round(12 * with_norms / 1e6, 1) == float(g["twelve layers approx M"])
    send = formulas.ring_volume_per_rank(block, int(g["R"])) * 2
    assert round(float(send) / 1e6, 1) == float(g["allgather send per GPU MB approx"])


# ---------------------------------------------------------------------------
# brute force and invariants
# ---------------------------------------------------------------------------

def check_rank_rows_bruteforce():
    for d0 in range(0, 41):
        rows = list(range(d0))
        for R in range(1, 10):
            seen = []
            for r in range(R):
                L = oracle.layout(oracle.PER_PARAM, R, [(d0, 3)])
                s, cnt = L.rank_rows(0, r)
                mine = brute.shard_dim0(rows, R, r)
                assert cnt == len(mine), (d0, R, r)
                if cnt:
                    assert mine == list(range(s, s + cnt))
                seen.extend(mine)
            assert seen == rows, (d0, R)          # disjoint, ordered, covering


def check_pack_matches_slicing_and_gather_restores():
    rng = np.random.default_rng(11)
    for trial in range(60):
        shapes = _tiny_shapes(rng)
        R = int(rng.integers(1, 7))
        numels = [int(np.prod(s)) for s in shapes]
        P = sum(numels)
        full = np.arange(1, P + 1, dtype=np.float32)
        params = []
        base = 0
        for n in numels:
            params.append(list(range(base + 1, base + n + 1)))
            base += n
        for mode in (oracle.PER_PARAM, oracle.FLAT):
            L = oracle.layout(mode, R, shapes)
            masters, p16 = oracle.pack(L, full, with_bf16=True)
            if mode == oracle.PER_PARAM:
                per_rank = brute.per_param_shards(params, shapes, R)
                for r in range(R):
                    expect = []
                    for i, sl in enumerate(per_rank[r]):
                        seg = [x for row in sl for x in row]
                        width = int(L.shard_rows[i]) * int(L.inner[i])
                        width = -(-width // oracle.SEG_ALIGN) * oracle.SEG_ALIGN
                        expect += seg + [0] * (width - len(seg))
                    assert masters[r].tolist() == expect, (shapes, R, r)
            else:
                pieces = brute.flat_shards(params, R)
                for r in range(R):
                    assert masters[r].tolist() == pieces[r], (shapes, R, r)
                assert brute.flat_gather(pieces, P) == full.tolist()
            for out in oracle.all_gather(L, masters):
                assert np.array_equal(out.view(np.uint32), full.view(np.uint32))
            for out in oracle.all_gather(L, p16):
                assert np.array_equal(out, oracle.f32_to_bf16(full))


def check_owner_matches_brute_force_and_gather():
    """The owner of every unit element is the rank whose brute-force slice
    holds it, and the gather reads exactly that shard slot."""
    rng = np.random.default_rng(17)
    for trial in range(60):
        shapes = _tiny_shapes(rng)
        R = int(rng.integers(1, 8))
        P = sum(int(np.prod(s)) for s in shapes)
        if P == 0:
            continue
        for mode in (oracle.PER_PARAM, oracle.FLAT):
            L = oracle.layout(mode, R, shapes)
            rank, index = oracle.owner(L, np.arange(P))
            if mode == oracle.PER_PARAM:
                ranges = brute.per_param_owner_ranges(shapes, R)
            else:
                S = L.shard_numel
                ranges = [[(min(r * S, P), min((r + 1) * S, P))] for r in range(R)]
            for r in range(R):
                mine = [j for a, b in ranges[r] for j in range(a, b)]
                assert np.flatnonzero(rank == r).tolist() == mine
            # tag every shard slot with (rank, slot) and gather
            shards = [(np.arange(L.shard_numel) + 1000 * r + 1).astype(np.float32)
                      for r in range(R)]
            full = oracle.all_gather(L, shards)[0]
            want = np.array([shards[r][i] for r, i in zip(rank, index)], np.float32)
            assert np.array_equal(full, want)


def check_reduce_scatter_integer_sums():
    """Integer-valued gradients sum exactly in any order: the oracle's shard
    times R equals the brute-force sum for power-of-two R, and is within one
    rounding of sum/R otherwise."""
    rng = np.random.default_rng(5)
    for trial in range(60):
        shapes = _tiny_shapes(rng)
        R = int(rng.integers(1, 10))
        P = sum(int(np.prod(s)) for s in shapes)
        gi = [rng.integers(-100, 101, P) for _ in range(R)]
        for mode in (oracle.PER_PARAM, oracle.FLAT):
            L = oracle.layout(mode, R, shapes)
            if mode == oracle.PER_PARAM:
                ranges = brute.per_param_owner_ranges(shapes, R)
            else:
                S = L.shard_numel
                ranges = [[(min(r * S, P), min((r + 1) * S, P))] for r in range(R)]
            sums = brute.reduce_scatter_sum([list(map(int, x)) for x in gi], R, ranges)
            for gdt in ("f32", "bf16"):
                grads = [x.astype(np.float32) for x in gi]
                if gdt == "bf16":
                    grads = [oracle.f32_to_bf16(x) for x in grads]
                gsh = oracle.reduce_scatter(L, grads)
                for r in range(R):
                    if mode == oracle.PER_PARAM:
                        got = np.concatenate([_owned(L, r, i, gsh[r]) for i in range(len(shapes))]
                                             ) if shapes else np.zeros(0, np.float32)
                        pad_mask = np.ones(L.shard_numel, bool)
                        for i in range(len(shapes)):
                            o = int(L.shard_off[i])
                            pad_mask[o:o + _owned(L, r, i, gsh[r]).size] = False
                        assert not gsh[r][pad_mask].any()
                    else:
                        got = gsh[r][:L.rank_numel(r)]
                        assert not gsh[r][L.rank_numel(r):].any()
                    assert len(got) == len(sums[r])
                    for x, s in zip(got.tolist(), sums[r]):
                        exact = Fraction(s, R)
                        if R in (1, 2, 4, 8):
                            assert Fraction(x) == exact
                        else:
                            assert abs(Fraction(x) - exact) <= abs(exact) * Fraction(1, 2 ** 22)


def check_reduce_scatter_is_allreduce_then_slice():
    """RS on rank r == segment r of (all-reduce of the rank gradients),
    the all-reduce done on whole buffers by numpy in the same rank order."""
    rng = np.random.default_rng(9)
    for trial in range(40):
        shapes = _tiny_shapes(rng)
        R = int(rng.integers(2, 9))
        P = sum(int(np.prod(s)) for s in shapes)
        for gdt in ("f32", "bf16"):
            gf = [rng.standard_normal(P).astype(np.float32) * np.float32(10.0 ** rng.integers(-3, 4))
                  for _ in range(R)]
            grads = gf if gdt == "f32" else [oracle.f32_to_bf16(x) for x in gf]
            widened = [x if gdt == "f32" else oracle.bf16_to_f32(x) for x in grads]
            allreduce = widened[0].copy()
            for q in range(1, R):
                allreduce = allreduce + widened[q]
            allreduce = allreduce * (np.float32(1) / np.float32(R))
            L = oracle.layout(oracle.PER_PARAM, R, shapes)
            gsh = oracle.reduce_scatter(L, grads)
            ranges = brute.per_param_owner_ranges(shapes, R)
            for r in range(R):
                got = np.concatenate([_owned(L, r, i, gsh[r]) for i in range(len(shapes))])
                want = np.concatenate([allreduce[a:b] for a, b in ranges[r]] or
                                      [np.zeros(0, np.float32)])
                assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def check_all_reduce_is_gather_of_reduce_scatter():
    """All-reduce == all-gather of the reduce-scatter shards, bit for bit, in
    both layouts ("FSDP2 的参数全聚合、梯度归约分片与显存峰值", §09; "从源码理解
    FSDP", §2.3: reduce-scatter equals all-reduce followed by taking segment
    r); and with integer gradients the all-reduce is the exact average."""
    rng = np.random.default_rng(23)
    for trial in range(40):
        shapes = _tiny_shapes(rng)
        R = int(rng.integers(1, 9))
        P = sum(int(np.prod(s)) for s in shapes)
        gf = [rng.standard_normal(P).astype(np.float32) for _ in range(R)]
        for gdt in ("f32", "bf16"):
            grads = gf if gdt == "f32" else [oracle.f32_to_bf16(x) for x in gf]
            ar = oracle.all_reduce(grads, out_bf16=False)
            for d in range(1, R):
                assert np.array_equal(ar[d].view(np.uint32), ar[0].view(np.uint32))
            ar16 = oracle.all_reduce(grads, out_bf16=True)
            assert np.array_equal(ar16[R - 1], oracle.f32_to_bf16(ar[0]))
            for mode in (oracle.PER_PARAM, oracle.FLAT):
                L = oracle.layout(mode, R, shapes)
                gathered = oracle.all_gather(L, oracle.reduce_scatter(L, grads))
                for d in range(R):
                    assert np.array_equal(gathered[d].view(np.uint32), ar[0].view(np.uint32))
        gi = [rng.integers(-64, 65, P) for _ in range(R)]
        ar = oracle.all_reduce([x.astype(np.float32) for x in gi], out_bf16=False)
        for j in range(P):
            exact = Fraction(int(sum(int(x[j]) for x in gi)), R)
            if R in (1, 2, 4, 8):
                assert Fraction(float(ar[0][j])) == exact
            else:
                assert abs(Fraction(float(ar[0][j])) - exact) <= abs(exact) * Fraction(1, 2 ** 22)


def check_accumulation_is_the_micro_batch_sum():
    """K micro-batches of integer gradients accumulate to their exact sum;
    the reduce-scatter of the accumulators equals the brute-force sum over
    micro-batches and ranks divided by R; the first micro-batch is copied,
    not added to zero, so -0 survives; accumulation is in micro-batch order
    (checked with values where the order changes the fp32 result)."""
    rng = np.random.default_rng(29)
    for trial in range(20):
        shapes = _tiny_shapes(rng)
        R = int(rng.integers(1, 6))
        K = int(rng.integers(1, 5))
        P = sum(int(np.prod(s)) for s in shapes)
        micro = [[rng.integers(-60, 61, P) for _ in range(R)] for _ in range(K)]
        for gdt in ("f32", "bf16"):
            acc = [np.zeros(P, np.float32) for _ in range(R)]
            for k in range(K):
                gk = [x.astype(np.float32) for x in micro[k]]
                if gdt == "bf16":
                    gk = [oracle.f32_to_bf16(x) for x in gk]
                oracle.accumulate(acc, gk, first=(k == 0))
            for q in range(R):
                want = sum(micro[k][q] for k in range(K))
                assert np.array_equal(acc[q], want.astype(np.float32))
            L = oracle.layout(oracle.PER_PARAM, R, shapes)
            gsh = oracle.reduce_scatter(L, acc)
            ranges = brute.per_param_owner_ranges(shapes, R)
            tot = [[int(sum(micro[k][q][j] for k in range(K))) for j in range(P)] for q in range(R)]
            sums = brute.reduce_scatter_sum(tot, R, ranges)
            for r in range(R):
                got = np.concatenate([_owned(L, r, i, gsh[r]) for i in range(len(shapes))])
                for x, sm in zip(got.tolist(), sums[r]):
                    exact = Fraction(sm, R)
                    if R in (1, 2, 4):
                        assert Fraction(x) == exact
                    else:
                        assert abs(Fraction(x) - exact) <= abs(exact) * Fraction(1, 2 ** 22)
    acc = [np.zeros(2, np.float32)]
    oracle.accumulate(acc, [np.array([-0.0, 5.0], np.float32)], first=True)
    assert np.signbit(acc[0][0]) and acc[0][1] == 5.0
    # (1 + 2^-24) + 2^-24 rounds differently from 1 + (2^-24 + 2^-24)
    e = np.float32(2.0 ** -24)
    acc = [np.zeros(1, np.float32)]
    for k, x in enumerate([np.float32(1.0), e, e]):
        oracle.accumulate(acc, [np.array([x], np.float32)], first=(k == 0))
    assert acc[0][0] == (np.float32(1.0) + e) + e


def check_zero3_inter_tensor_layout():
    """ZeRO-3 inter-tensor sharding ("从源码理解 FSDP", §2.1 and its table):
    every tensor lives whole on one owner; owners follow the brute-force
    partition; gather(pack(W)) == W; the reduce-scatter leaves each tensor's
    rank-averaged gradient on its owner only (== all-reduce, then the owner's
    tensors); and on the page's own 512/8/2048 block the load is uneven,
    while the FSDP layout gives every rank the same 786,432."""
    rng = np.random.default_rng(37)
    for trial in range(50):
        shapes = _tiny_shapes(rng, max_params=6)
        R = int(rng.integers(1, 6))
        numels = [int(np.prod(s)) for s in shapes]
        P = sum(numels)
        L = oracle.layout(oracle.ZERO3, R, shapes)
        parts = brute.zero3_parts(numels, R)
        for r, idx in enumerate(parts):
            for i in idx:
                assert int(L.owner[i]) == r
        for i in range(len(shapes)):
            held = [L.rank_rows(i, r)[1] for r in range(R)]
            assert sorted(held)[-1] == shapes[i][0] and sum(held) == shapes[i][0]
        full = np.arange(1, P + 1, dtype=np.float32)
        masters, p16 = oracle.pack(L, full, with_bf16=True)
        for out in oracle.all_gather(L, masters):
            assert np.array_equal(out, full)
        base = np.cumsum([0] + numels)
        for r in range(R):   # a rank's buffer holds exactly its tensors, padded
            want = []
            for i in parts[r]:
                seg = list(range(base[i] + 1, base[i] + numels[i] + 1))
                want += seg + [0] * (-(-numels[i] // oracle.SEG_ALIGN) * oracle.SEG_ALIGN
                                     - numels[i])
            want += [0] * (L.shard_numel - len(want))
            assert masters[r].tolist() == want
        grads = [rng.standard_normal(P).astype(np.float32) for _ in range(R)]
        ar = oracle.all_reduce(grads, out_bf16=False)[0]
        gsh = oracle.reduce_scatter(L, grads)
        for r in range(R):
            got = np.concatenate([_owned(L, r, i, gsh[r]) for i in range(len(shapes))])
            want = np.concatenate([ar[base[i]:base[i] + numels[i]] for i in parts[r]] or
                                  [np.zeros(0, np.float32)])
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
        rank, index = oracle.owner(L, np.arange(P)) if P else (np.zeros(0), np.zeros(0))
        for i in range(len(shapes)):
            assert np.all(rank[base[i]:base[i + 1]] == L.owner[i])
    g = golden("block_sharding.txt")
    R = int(g["R"])
    shapes = [s for _, s in _matrices_only()]
    Z = oracle.layout(oracle.ZERO3, R, shapes)
    F = oracle.layout(oracle.PER_PARAM, R, shapes)
    loads = [Z.rank_numel(r) for r in range(R)]
    assert sum(loads) == int(g["fsdp1 flat length"])
    assert [F.rank_numel(r) for r in range(R)] == [int(g["fsdp2 total per GPU"])] * R
    assert max(loads) > int(g["fsdp2 total per GPU"])


def check_reduce_scatter_special_cases():
    # R = 1: the shard is the gradient itself
    g = np.array([1.5, -2.25, 3e-8, -0.0], np.float32)
    L = oracle.layout(oracle.PER_PARAM, 1, [(4,)])
    out = oracle.reduce_scatter(L, [g])[0][:4]
    assert np.array_equal(out.view(np.uint32), g.view(np.uint32))
    # the fold starts from rank 0's value, so (-0) + (-0) stays -0
    L2 = oracle.layout(oracle.PER_PARAM, 2, [(2,)])
    z = np.array([-0.0, -0.0], np.float32)
    out = oracle.reduce_scatter(L2, [z, z])
    assert np.signbit(out[0][0]) and np.signbit(out[1][0])
    # the average is a multiply by fl(1/R): for R = 3 pick sums where that
    # differs from a correctly rounded division and check the multiply wins
    third = np.float32(1) / np.float32(3)
    xs = np.arange(1, 4000, dtype=np.float32) * np.float32(1.0009765625)
    differs = xs[(xs * third) != (xs / np.float32(3))][:8]
    assert differs.size > 0
    L3 = oracle.layout(oracle.PER_PARAM, 3, [(differs.size * 3,)])
    zeros = np.zeros(differs.size * 3, np.float32)
    g0 = np.tile(differs, 3)
    out = oracle.reduce_scatter(L3, [g0, zeros, zeros])
    got = out[0][:differs.size]
    assert np.array_equal(got, differs * third)


# ---------------------------------------------------------------------------
# AdamW
# ---------------------------------------------------------------------------

def check_adamw_closed_form_first_step():
    """At t = 1 from m = v = 0: m_hat = g and v_hat = g^2, so
    w1 = w0 (1 - lr wd) - lr g / (|g| + eps)."""
    rng = np.random.default_rng(2)
    for scale in (1.0, 1e-3, 1e-7):
        g = (rng.standard_normal(256) * scale).astype(np.float32)
        w = rng.standard_normal(256).astype(np.float32)
        m = np.zeros_like(w)
        v = np.zeros_like(w)
        w0 = w.astype(np.float64)
        gd = g.astype(np.float64)
        oracle.adamw(g.copy(), w, m, v, HP, 1)
        expect = w0 * (1 - HP.lr * HP.weight_decay) - HP.lr * gd / (np.abs(gd) + HP.eps)
        assert np.all(np.abs(w - expect) <= 4e-7 * np.maximum(1, np.abs(expect)))
        assert np.allclose(m, (1 - HP.beta1) * gd, rtol=1e-6, atol=0)
        assert np.allclose(v, (1 - HP.beta2) * gd * gd, rtol=1e-5, atol=0)


def check_adamw_matches_torch():
    """Several steps against torch.optim.AdamW on CPU (a library routine),
    for ordinary, tiny (eps-dominated) and outlier gradients."""
    import torch
    rng = np.random.default_rng(4)
    for scale, wd in ((1.0, 0.01), (1e-6, 0.01), (1e4, 0.1), (1e-3, 0.0)):
        hp = oracle.AdamWHP(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=wd)
        n = 128
        w = rng.standard_normal(n).astype(np.float32)
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
        p = torch.nn.Parameter(torch.from_numpy(w.copy()))
        opt = torch.optim.AdamW([p], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                                weight_decay=hp.weight_decay, foreach=False)
        for t in range(1, 7):
            g = (rng.standard_normal(n) * scale).astype(np.float32)
            # re-sync the state each step: the bound is per step
            with torch.no_grad():
                p.copy_(torch.from_numpy(w))
            if t > 1:
                st = opt.state[p]
                st["exp_avg"].copy_(torch.from_numpy(m))
                st["exp_avg_sq"].copy_(torch.from_numpy(v))
            p.grad = torch.from_numpy(g.copy())
            opt.step()
            # m combines two terms that can cancel, so its bound is set by
            # their size; v adds two non-negative terms
            m_scale = np.abs(m) + np.abs(g)
            oracle.adamw(g, w, m, v, hp, t)
            ref = p.detach().numpy()
            st = opt.state[p]
            assert np.all(np.abs(w - ref) <= 1e-5 * np.maximum(1, np.abs(ref))), (scale, t)
            ea, eq = st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
            assert np.all(np.abs(m - ea) <= 1e-6 * m_scale), (scale, t)
            assert np.all(np.abs(v - eq) <= 1e-5 * np.abs(eq)), (scale, t)


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------

def check_bf16_round_to_nearest_even():
    """fp32 -> bf16 against torch's conversion (a library routine) on every
    upper half with the rounding-critical lower halves, plus random bits."""
    import torch
    hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xC000, 0xFFFF], np.uint32)
    bits = (hi[:, None] | lows[None, :]).ravel()
    bits = np.concatenate([bits, np.random.default_rng(1).integers(0, 1 << 32, 1 << 20,
                                                                     dtype=np.uint32)])
    x = bits.view(np.float32)
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(oracle.bf16_to_f32(ours[nan])))
    # widening is exact and narrowing a bf16 value is the identity
    every = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    wide = oracle.bf16_to_f32(every)
    ok = ~np.isnan(wide)
    assert np.array_equal(oracle.f32_to_bf16(wide)[ok], every[ok])


def exhaustive_bf16_rounding():
    """fp32 -> bf16 narrowing against torch's conversion on all 2^32 bit
    patterns (NaNs: both NaN). Kept out of ALL_CHECKS, which the mutation
    test runs once per planted mistake; check_bf16_round_to_nearest_even
    covers the rounding-critical patterns there."""
    import torch
    chunk = 1 << 26
    for c in range((1 << 32) // chunk):
        bits = np.arange(c * chunk, (c + 1) * chunk, dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        ours = oracle.f32_to_bf16(x)
        ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(x)
        assert np.array_equal(ours[~nan], ref[~nan]), c
        assert np.all(np.isnan(oracle.bf16_to_f32(ours[nan]))), c


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
