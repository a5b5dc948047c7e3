"""Host logic of the GEMMs' split-K planner (no GPU needed).

The library splits the contraction of some output tiles (128 x 256) when the
persistent launch's last wave would leave many of the 148 SMs idle.  These
tests pin the plans of the workloads' products and the planner's invariants
over a sweep of shapes."""
import math

import pytest

from fp8_block_scaled_16_b300 import binding as B

SMS = 148
FLAG_BYTES = 64 * 1024
PARTIAL_BYTES = 128 * 256 * 4


def tiles_of(rows, cols):
    return math.ceil(rows / 128) * math.ceil(cols / 256)


def plan(tiles, kblocks, sms=SMS):
    return B.fp8bs_debug_split_plan(tiles, kblocks, sms)


def test_short_contraction_is_not_split():
    """Attention QKV forward at 8192 tokens: 64 x 12 = 768 tiles = 5 full
    waves + 28 tiles of 16 K blocks.  Splitting the 28 would save at most
    12 blocks of the last wave, less than moving their FP32 partials costs
    (each part's publication ~5 blocks, ~2 per partial for the last part's sum)."""
    p = plan(tiles_of(8192, 3072), 2048 // 128)
    assert p == {"splits": 1, "tail_first": 0, "units": 768, "bytes": 0}


def test_long_contraction_tail_is_split():
    """The same 768 tiles with a 64-block contraction: the 28 tiles past the
    5 full waves are split in 5 parts (5 x 28 = 140 units <= 148 SMs); every
    part publishes its partial (5 per split tile)."""
    p = plan(768, 64)
    assert p == {"splits": 5, "tail_first": 740, "units": 740 + 5 * 28,
                 "bytes": FLAG_BYTES + 5 * 28 * PARTIAL_BYTES}


@pytest.mark.parametrize("rows,cols,kblocks,splits,first", [
    (3072, 2048, 256, 3, 148),   # QKV weight gradient at 32768 tokens: 192 tiles
    (2048, 5632, 256, 2, 296),   # down-projection weight gradient: 352 tiles
    (2048, 2048, 256, 1, 0),     # O weight gradient: 128 tiles in one wave, nothing to gain
    (11264, 2048, 256, 1, 0),    # gate+up weight gradient: 704 tiles, last wave 76% full
    (32768, 11264, 16, 1, 0),    # gate+up forward: 11264 tiles, the tail is 1% of the work
    (16384, 2048, 88, 1, 0),     # gate+up data gradient at 16384 tokens
    (2432, 2048, 32, 4, 148),    # 152 tiles: the 4 past one full wave in 4 parts of 8 blocks
    (3968, 2048, 128, 4, 0),     # 248 tiles (1.7 waves): every tile in 4 parts
])
def test_workload_plans(rows, cols, kblocks, splits, first):
    p = plan(tiles_of(rows, cols), kblocks)
    assert (p["splits"], p["tail_first"]) == (splits, first)
    if splits == 1:
        assert p["bytes"] == 0 and p["units"] == tiles_of(rows, cols)


def wave_time(units_by_len, sms):
    """Makespan of units taken round-robin by persistent CTAs in index
    order, each costing its K blocks + 1 (a direct simulation, independent
    of the planner's closed-form estimate)."""
    load = [0.0] * sms
    for i, k in enumerate(units_by_len):
        load[i % sms] += k + 1
    return max(load)


@pytest.mark.parametrize("sms", [148, 132, 7])
def test_plan_invariants_over_a_sweep(sms):
    for tiles in list(range(1, 40)) + [147, 148, 149, 151, 190, 296, 300, 767, 768, 769, 2817]:
        for kblocks in (1, 3, 4, 8, 16, 17, 44, 88, 256):
            p = plan(tiles, kblocks, sms)
            s, first, units = p["splits"], p["tail_first"], p["units"]
            if s == 1:
                assert (first, units, p["bytes"]) == (0, tiles, 0)
                continue
            split_tiles = tiles - first
            assert 0 <= first < tiles and units == first + s * split_tiles
            assert p["bytes"] == FLAG_BYTES + s * split_tiles * PARTIAL_BYTES
            assert split_tiles * 8 * 8 <= FLAG_BYTES   # one 8-byte arrival counter per tile slice
            if first == 0:
                assert 2 <= s <= 4 and kblocks // s >= 16
            else:
                assert first % sms == 0 and s * split_tiles <= sms and kblocks // s >= 4
            # The split schedule is really shorter: simulate both.
            # Units in the kernel's order: whole tiles, then part 0 of the
            # split tiles, part 1, ...
            parts = [(j * kblocks) // s for j in range(s + 1)]
            lens = [kblocks] * first
            for j in range(s):
                lens += [parts[j + 1] - parts[j]] * split_tiles
            assert wave_time(lens, sms) < wave_time([kblocks] * tiles, sms)


def test_rejects_bad_arguments():
    for args in ((0, 16, SMS), (10, 0, SMS), (10, 16, 0), (-1, 16, SMS)):
        with pytest.raises(B.Fp8bsError):
            plan(*args)
