"""Pins for the oracle's quantizers (CPU only): hand-derived tiles, the
invariants the scheme implies, and identities between the three layouts."""
import numpy as np
import torch

import oracle
from fp8_block_scaled_16_b300 import inputs


def bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def f32(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.float32).numpy()


def test_hand_tile_amax_448_is_identity_scale():
    # amax = 448 -> s = 448/448 = 1, inv = 1: payloads are the E4M3 codes of
    # the (exactly representable) values themselves.
    vals = [448.0, -448.0, 1.0, -1.0, 3.0, 6.0, 0.5, 2.0 ** -9, 0.0, -0.0, 240.0, 256.0]
    codes = [0x7E, 0xFE, 0x38, 0xB8, 0x44, 0x4C, 0x30, 0x01, 0x00, 0x80, 0x77, 0x78]
    row = np.zeros(128, np.float32)
    row[: len(vals)] = vals
    q, s = oracle.quant_rowwise_1x128(bf16(row[None, :]))
    assert s.shape == (1, 128) and s[0, 0] == 1.0      # one row, padded to a 128-token block
    assert list(q[0, : len(codes)]) == codes
    assert np.all(q[0, len(codes):] == 0)


def test_hand_tile_amax_224_scales_by_two():
    # amax = 224 -> s = 0.5, inv = 2: 224 -> 448 (0x7E), 1 -> 2 (0x40),
    # -3 -> -6 (0xCC), 0.75 -> 1.5 (0x3C).
    row = np.zeros(128, np.float32)
    row[:4] = [224.0, 1.0, -3.0, 0.75]
    q, s = oracle.quant_rowwise_1x128(bf16(row[None, :]))
    assert s[0, 0] == 0.5
    assert list(q[0, :4]) == [0x7E, 0x40, 0xCC, 0x3C]


def test_all_zero_tile():
    x = torch.zeros(2, 256, dtype=torch.bfloat16)
    x[1, :128] = -0.0
    q, s = oracle.quant_rowwise_1x128(x)
    assert np.all(s == 1.0)
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0x80) and np.all(q[1, 128:] == 0)


def test_tiny_tile_clamps_reciprocal():
    # amax = 2^-133 (smallest BF16 subnormal): 448/amax overflows FP32, so the
    # multiplier is clamped to FLT_MAX = 2^128 (1 - 2^-24); zeros stay zero
    # (no 0*Inf NaN), the amax element becomes 2^-5 (1 - 2^-24), which rounds
    # to 2^-5 (code 0x10, here negative: 0x90), and the stored scale is still
    # amax/448.
    row = np.zeros(128, np.float32)
    row[5] = -(2.0 ** -133)
    q, s = oracle.quant_rowwise_1x128(bf16(row[None, :]))
    assert q[0, 5] == 0x90 and np.all(np.delete(q[0], 5) == 0)
    assert s[0, 0] == np.float32(2.0 ** -133) / np.float32(448.0)
    assert s[0, 0] > 0


def test_scale_is_amax_over_448_and_amax_element_maps_to_448():
    x = inputs.random_bf16((64, 512), seed=11, std=3.0)
    x[3, 7] = 1e4
    q, s = oracle.quant_rowwise_1x128(x)
    xf = f32(x).reshape(64, 4, 128)
    amax = np.abs(xf).max(axis=2).astype(np.float32)          # [rows][blocks]
    assert np.array_equal(s[:, :64], (amax / np.float32(448.0)).T)    # IEEE float32 division
    assert np.all(s[:, 64:] == 1.0)                           # padding tokens: all-zero tiles
    qb = q.reshape(64, 4, 128)
    is_max = np.abs(xf) == amax[:, :, None]
    assert np.all((qb[is_max] & 0x7F) == 0x7E)
    assert np.all((qb & 0x7F) <= 0x7E)                        # never NaN


def test_power_of_two_equivariance():
    x = inputs.random_bf16((32, 256), seed=12)
    q0, s0 = oracle.quant_rowwise_1x128(x)
    for j in (-7, -1, 1, 5):
        q1, s1 = oracle.quant_rowwise_1x128(x * (2.0 ** j))
        assert np.array_equal(q0, q1)
        assert np.array_equal(s1[:, :32], s0[:, :32] * np.float32(2.0 ** j))


def test_dequantization_error_bound():
    x = inputs.random_bf16((128, 1024), seed=13, std=2.0)
    x[:, 17] *= 80.0
    q, s = oracle.quant_rowwise_1x128(x)
    deq = oracle.e4m3_decode(q).reshape(128, 8, 128) * s.T[:, :, None].astype(np.float64)
    xf = f32(x).astype(np.float64).reshape(128, 8, 128)
    err = np.abs(deq - xf)
    scaled = np.abs(xf) / s.T[:, :, None]                    # |x| * 448 / amax
    normal = scaled >= 2.0 ** -6
    # 3 mantissa bits: half an ulp is 2^-4 of the value; subnormal step 2^-9
    # times the scale.  (1 + 2^-20) covers the rounding of s and 448/amax.
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(xf[normal]) * (1 + 2.0 ** -20))
    sub = ~normal
    bound = (2.0 ** -10 * np.broadcast_to(s.T[:, :, None], xf.shape)[sub]) * (1 + 2.0 ** -20)
    assert np.all(err[sub] <= bound)


def test_colwise_is_rowwise_of_transpose():
    x = inputs.random_bf16((384, 256), seed=14)
    x[:, 9] *= 40.0
    qT, sT = oracle.quant_colwise_128x1_T(x)
    q_r, s_r = oracle.quant_rowwise_1x128(x.t().contiguous())
    assert qT.shape == (256, 384) and sT.shape == (3, 256)
    assert np.array_equal(qT, q_r)
    assert np.array_equal(sT, s_r)


def test_weight_blocks_transpose_and_scales():
    w = inputs.random_bf16((384, 256), seed=15, std=0.02)
    w[200, 3] = 0.9
    q, qT, s = oracle.quant_weight_128x128(w)
    assert np.array_equal(qT, q.T)
    wf = f32(w).reshape(3, 128, 2, 128)
    amax = np.abs(wf).max(axis=(1, 3)).astype(np.float32)
    assert np.array_equal(s, amax / np.float32(448.0))
    # A block whose amax equals a 1x128 row tile's amax quantizes that row
    # exactly like the row-wise quantizer does.
    q_row, _ = oracle.quant_rowwise_1x128(w)
    blk = (1, 0)  # block rows 128..255, cols 0..127 holds w[200,3] = 0.9, its amax
    r = 200
    assert abs(float(wf[1, 72, 0, 3])) == amax[blk]
    assert np.array_equal(q[r, :128], q_row[r, :128])
    assert np.array_equal(q[r - 128 + 128, :128], q_row[r, :128])


def test_token_tail_equals_zero_padding():
    """Reading for token counts that are not a multiple of 128: the last
    128x1 tile covers the tokens present and the padding tokens count as
    zeros.  So quantizing 300 tokens must equal quantizing the same tensor
    padded with zero tokens to 384 (row scales of padding rows are 1, the
    padding payload is 0x00), and the partial tile's scale is numpy's amax of
    the present tokens / 448."""
    M, K = 300, 256
    x = inputs.random_bf16((M, K), seed=16)
    x[:, 3] *= 30.0
    xp = torch.zeros(384, K, dtype=torch.bfloat16)
    xp[:M] = x
    q, s = oracle.quant_rowwise_1x128(x)
    qp, sp = oracle.quant_rowwise_1x128(xp)
    assert q.shape == (M, K) and s.shape == (2, 384)
    assert np.array_equal(q, qp[:M])
    assert np.array_equal(s[:, :M], sp[:, :M]) and np.all(s[:, M:] == 1.0)
    qT, sT = oracle.quant_colwise_128x1_T(x)
    qTp, sTp = oracle.quant_colwise_128x1_T(xp)
    assert qT.shape == (K, 384) and sT.shape == (3, K)
    assert np.array_equal(qT, qTp) and np.array_equal(sT, sTp)
    assert np.all(qT[:, M:] == 0)
    tail_amax = np.abs(f32(x[256:])).max(axis=0).astype(np.float32)     # 44 tokens
    assert np.array_equal(sT[2], tail_amax / np.float32(448.0))


def test_token_tail_gemm_rows_do_not_depend_on_padding():
    M, N, K = 300, 256, 256
    x = inputs.random_bf16((M, K), seed=17)
    w = inputs.random_bf16((N, K), seed=18, std=0.02)
    xq, sx = oracle.quant_rowwise_1x128(x)
    wq, _, sw = oracle.quant_weight_128x128(w, want_t=False)
    acc, y, _ = oracle.gemm_fprop(xq, sx, wq, sw)
    xp = torch.zeros(384, K, dtype=torch.bfloat16)
    xp[:M] = x
    xqp, sxp = oracle.quant_rowwise_1x128(xp)
    accp, yp, _ = oracle.gemm_fprop(xqp, sxp, wq, sw)
    assert acc.shape == (M, N)
    assert np.array_equal(acc, accp[:M]) and np.array_equal(y, yp[:M])
    assert not accp[M:].any()
