"""Host logic of the GEMMs' tile order (no GPU needed).

The persistent CTAs take output tiles (128 x 256) in column strips; the
library picks the strip width whose estimated DRAM reads of operand panels
are smallest, simulating L2 reuse wave by wave.  These tests pin the choice
on the decoder layer's products at 32768 tokens and the estimate's
invariants; that the outputs do not depend on the order is covered by the
GPU parity tests of the same shapes."""
import math

import pytest

from fp8_block_scaled_16_b300 import binding as B

T = 32768
L2 = 126 << 20


def tiles(rows, cols):
    return math.ceil(rows / 128), math.ceil(cols / 256)


def order(rows, cols, kc, splits=1, first=0, grid=148, l2=L2, out_bytes=2):
    m, n = tiles(rows, cols)
    return m, n, B.fp8bs_debug_tile_order(m, n, kc, splits, first, grid, l2, out_bytes)


@pytest.mark.parametrize("rows,cols,kc", [
    (T, 3072, 2048),    # QKV forward
    (T, 11264, 2048),   # gate+up forward: strips would re-read X once per strip
    (T, 5632, 2048),    # down data gradient
    (T, 2048, 11264),   # gate+up data gradient
])
def test_short_contractions_stay_row_major_and_read_each_panel_once(rows, cols, kc):
    m, n, r = order(rows, cols, kc)
    assert r["strip"] == n
    assert r["dram_bytes"] == m * 128 * kc + n * 256 * kc


def test_down_projection_weight_gradient_goes_column_by_column():
    """2048 x 5632 over 32768 tokens, last 56 tiles split in 2: 8 MB panels
    do not survive in L2 from one wave to the next, so the order with the
    fewest distinct panels per wave (one column at a time) reads least."""
    m, n, r = order(2048, 5632, T, splits=2, first=296)
    assert r["strip"] == 1
    assert r["dram_bytes"] < 0.7 * r["row_major_dram_bytes"]


@pytest.mark.parametrize("rows,cols,kc,splits,first", [
    (3072, 2048, T, 3, 148), (2048, 2048, T, 1, 0), (11264, 2048, T, 1, 0), (2048, 5632, T, 2, 296),
    (T, 2048, 5632, 1, 0), (1000, 9000, 4096, 1, 0), (128, 256, 128, 1, 0),
])
def test_estimate_bounds(rows, cols, kc, splits, first):
    m, n, r = order(rows, cols, kc, splits, first)
    floor = m * 128 * kc + n * 256 * kc                 # every panel at least once
    units = m * n if splits == 1 else first + splits * (m * n - first)
    ceiling = math.ceil(units / 148) * (m * 128 * kc + n * 256 * kc)   # every panel every wave
    assert 1 <= r["strip"] <= n
    assert floor <= r["dram_bytes"] <= r["row_major_dram_bytes"] <= ceiling


def test_everything_fits_in_l2_reads_once_whatever_the_shape():
    # A huge L2: nothing is ever evicted, so the estimate is the floor and row-major is kept.
    for rows, cols, kc in ((2048, 5632, T), (11264, 2048, T), (4096, 4096, 8192)):
        m, n, r = order(rows, cols, kc, l2=1 << 40)
        assert r["strip"] == n and r["dram_bytes"] == m * 128 * kc + n * 256 * kc


def test_rejects_bad_arguments():
    good = dict(m_tiles=4, n_tiles=4, kc=1024, splits=1, tail_first=0, grid=148, l2_bytes=L2, out_bytes=2)
    for k, v in (("m_tiles", 0), ("n_tiles", -1), ("kc", 0), ("grid", 0), ("l2_bytes", 0), ("out_bytes", 3),
                 ("splits", 0)):
        with pytest.raises(B.Fp8bsError):
            B.fp8bs_debug_tile_order(**{**good, k: v})
    with pytest.raises(B.Fp8bsError):
        B.fp8bs_debug_tile_order(**{**good, "splits": 2, "tail_first": 16})
