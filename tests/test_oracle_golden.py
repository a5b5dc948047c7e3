"""The oracle's quantizers against hand-derived tiles stored in
tests/golden/quant_tiles.txt (CPU only).  The fixture's values come from the
E4M3 bit layout and the scale definition, worked by hand (derivations are in
the file); the scale bits are also re-derived here with numpy's IEEE FP32
division, independently of the oracle."""
import os

import numpy as np
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def load_cases():
    cases = []
    with open(os.path.join(HERE, "golden", "quant_tiles.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            layout, inp, sbits, fill, codes = [p.strip() for p in line.split("|")]
            vals = {int(k): float(v) for k, v in (e.split("=") for e in inp.split())}
            want = {int(k): int(v, 16) for k, v in (e.split("=") for e in codes.split())}
            cases.append((layout, vals, int(sbits, 16), int(fill, 16), want))
    return cases


def test_fixture_has_cases():
    assert len(load_cases()) >= 6


def test_oracle_matches_hand_derived_tiles():
    for layout, vals, sbits, fill, want in load_cases():
        tile = np.zeros(128, np.float32)
        for i, v in vals.items():
            tile[i] = v
        amax = np.float32(np.abs(tile).max())
        if amax > 0:  # the stored bits are the IEEE quotient amax/448
            assert int(np.array([amax / np.float32(448.0)]).view(np.uint32)[0]) == sbits
        xb = torch.from_numpy(tile).to(torch.bfloat16)
        assert torch.equal(xb.float(), torch.from_numpy(tile)), "fixture values must be exact in BF16"
        if layout == "row":
            q, s = oracle.quant_rowwise_1x128(xb[None, :])
            payload, scale = q[0], s[0, 0]
        else:
            x = torch.zeros(128, 128, dtype=torch.bfloat16)
            x[:, 3] = xb
            qT, sT = oracle.quant_colwise_128x1_T(x)
            payload, scale = qT[3], sT[0, 3]
        assert int(np.array([scale]).view(np.uint32)[0]) == sbits, (layout, vals)
        expect = np.full(128, fill, np.uint8)
        for i, c in want.items():
            expect[i] = c
        assert np.array_equal(payload, expect), (layout, vals, payload[:8])
