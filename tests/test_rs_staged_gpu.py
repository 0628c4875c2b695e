"""The reduce-scatter + AdamW kernel that stages the R gradient slices in
shared memory (bulk copies, a ring of stages per thread block), against the
oracle element by element.

The library takes it for R = 4, 8 with bf16 gradients and R = 2, 4 with fp32
gradients, on launches of at least 32 tiles (2,048 elements) per staged
thread block (2 per SM); smaller launches and other R take the register
kernel. The units here (24M parameters) clear that bar, and every block's
ring of stages wraps many times. FSDP2 dim-0 sharding of odd row widths puts
aligned rank pieces, whose tiles are staged, and misaligned pieces, whose
tiles take the register path inside the same kernel, into one launch; pieces
whose length is not a multiple of 8 end in partial vectors."""
import numpy as np
import pytest
import torch

from parity import UnitCase, run_unit_case, run_units_case

pytestmark = pytest.mark.gpu

TILE = 2048
MIN_TILES_PER_CTA = 32
CTAS_PER_SM = 2

# 24.1M parameters: one piece per rank of every tensor (FSDP2)
SHAPES = [(4096, 513), (3000, 1001), (2049, 64), (127,), (8192, 256), (16384, 1024)]


def _pieces(shapes, R):
    """(full start, shard start, length) of every non-empty FSDP2 rank piece."""
    full_off = shard_off = 0
    out = []
    for s in shapes:
        d0 = s[0]
        inner = int(np.prod(s[1:], dtype=np.int64)) if len(s) > 1 else 1
        rows = -(-d0 // R)
        for r in range(R):
            n = max(0, min(rows, d0 - r * rows)) * inner
            if n:
                out.append((full_off + r * rows * inner, shard_off, n))
        full_off += d0 * inner
        shard_off += rows * inner
    return out


def _staged_launch(shapes, R, units=1):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = units * sum(-(-n // TILE) for _, _, n in _pieces(shapes, R))
    return tiles >= MIN_TILES_PER_CTA * CTAS_PER_SM * sms


@pytest.mark.parametrize("R", [2, 4, 8])
def test_units_mix_staged_and_register_tiles(R):
    pieces = _pieces(SHAPES, R)
    aligned = sum(1 for f, s, _ in pieces if f % 8 == 0 and s % 8 == 0)
    assert 0 < aligned < len(pieces)
    assert any(n % 8 for _, _, n in pieces)


@pytest.mark.parametrize("R,grad_dtype,param_dtype", [
    (2, "f32", "f32"), (4, "bf16", "bf16"), (4, "f32", "bf16"),
    (8, "bf16", "f32"), (8, "bf16", "bf16"),
    # the register kernel at the same size, as controls: bf16 R = 2 (too few
    # gradient bytes to gain from staging), fp32 R = 8 (a stage over 32 KB)
    (2, "bf16", "bf16"), (8, "f32", "f32"),
])
def test_staged_unit_vs_oracle(cuda_lib, R, grad_dtype, param_dtype):
    assert _staged_launch(SHAPES, R)
    run_unit_case(UnitCase(shapes=SHAPES, R=R, param_dtype=param_dtype, grad_dtype=grad_dtype,
                           seed=40 + R, g_std=1e-3, outlier_frac=0.01, step=3,
                           prior_moments=True))


def test_staged_units_per_call_vs_oracle(cuda_lib):
    """Two units in one launch of the staged kernel (its multi-unit form)."""
    assert _staged_launch(SHAPES, 8, units=2)
    cases = [UnitCase(shapes=SHAPES, R=8, seed=60 + k) for k in range(2)]
    run_units_case(cases, step=2)


def test_flat_units_with_misaligned_rank_pieces(cuda_lib):
    """FSDP1 FlatParameter whose rank pieces start off the 8-element grid
    (P/R not a multiple of 8): every tile of ranks 1.. takes the register
    path inside the staged kernel, rank 0's tiles are staged."""
    shapes = [(24_000_003,), (999, 37)]
    P = sum(int(np.prod(s)) for s in shapes)
    S = -(-P // 4)
    assert S % 8 != 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 4 * -(-S // TILE) >= MIN_TILES_PER_CTA * CTAS_PER_SM * sms
    run_unit_case(UnitCase(shapes=shapes, R=4, mode="flat", seed=70, step=2,
                           prior_moments=True))


@pytest.mark.parametrize("mode,shapes", [
    ("flat", [(7_427_862,)]),                  # S odd: ranks 1-7 start off the 8-element grid
    ("per_param", [(4097, 513), (1001, 63), (5,)]),
])
def test_register_kernel_realigned_tiles_vs_oracle(cuda_lib, mode, shapes):
    """bf16 gradients at R = 8 on a launch too small to stage: the register
    kernel reads misaligned tiles with aligned 16-byte loads and realigns
    them in registers."""
    P = sum(int(np.prod(s)) for s in shapes)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert -(-P // TILE) + 8 * len(shapes) < MIN_TILES_PER_CTA * CTAS_PER_SM * sms
    run_unit_case(UnitCase(shapes=shapes, R=8, mode=mode, seed=90, step=2, outlier_frac=0.01,
                           prior_moments=True))


def test_bounded_wait_gives_up_and_the_device_stays_usable(cuda_lib):
    """The staged kernel's bounded wait, on an mbarrier that nothing
    completes: the block gives up, counts itself, and the device still runs
    a staged step correctly afterwards."""
    from fully_sharded_state_gb300 import fsdp_stage_wait_selftest, fsdp_stage_wait_timeouts
    assert fsdp_stage_wait_selftest() == 1
    assert fsdp_stage_wait_selftest() == 1
    assert fsdp_stage_wait_timeouts() == 0  # the real counter is untouched
    run_unit_case(UnitCase(shapes=SHAPES, R=8, seed=80, step=2))


def test_no_stage_wait_gave_up(cuda_lib):
    from fully_sharded_state_gb300 import fsdp_stage_wait_timeouts
    assert fsdp_stage_wait_timeouts() == 0
