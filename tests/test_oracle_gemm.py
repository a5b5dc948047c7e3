"""Pins for the oracle's block-scaled GEMMs (CPU only).

Every E4M3 value is an integer multiple of 2^-9, so an integer matrix product
of the codes' values times 512 gives each 128-block's exact partial sum P_b.
From there the promotion chain acc = fma(P_b, sa*sb, acc) is emulated in
exact rational arithmetic with a correctly rounded FP32 step, independently
of the C oracle.
"""
from fractions import Fraction

import numpy as np
import torch

import oracle
from fp8_block_scaled_16_b300 import inputs


def rn_f32(v: Fraction) -> float:
    """Round a rational to the nearest FP32 value, ties to even (normal and
    subnormal results; no overflow in these tests)."""
    if v == 0:
        return 0.0
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)                       # subnormal spacing below 2^-126
    ulp = Fraction(2) ** (e - 23)
    q, r = divmod(a, ulp)
    q = int(q)
    if r > ulp / 2 or (r == ulp / 2 and q % 2 == 1):
        q += 1
    return sign * float(q * ulp)


def random_codes(shape, rng) -> np.ndarray:
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3F                  # no NaN payloads
    return c


def int_values(codes: np.ndarray) -> np.ndarray:
    """Decoded E4M3 values times 512, as exact int64 (via the decoder)."""
    v = oracle.e4m3_decode(codes) * 512.0
    assert np.all(v == np.round(v))
    return v.astype(np.int64)


def block_partials(a_codes, b_codes):
    """P_b * 2^18 for every output and 128-block: [rows][cols][blocks] int64."""
    ia, ib = int_values(a_codes), int_values(b_codes)
    kb = a_codes.shape[1] // 128
    return np.stack([ia[:, j * 128:(j + 1) * 128] @ ib[:, j * 128:(j + 1) * 128].T
                     for j in range(kb)], axis=2)


def emulate_promotion(P, sa, sb):
    """acc = fma(f32(P_b), f32(sa_b*sb_b), acc) over blocks, exactly rounded."""
    acc = 0.0
    for j in range(P.shape[0]):
        p32 = rn_f32(Fraction(int(P[j]), 2 ** 18))
        s32 = float(np.float32(sa[j]) * np.float32(sb[j]))   # IEEE float32 product
        acc = rn_f32(Fraction(p32) * Fraction(s32) + Fraction(acc))
    return acc


def test_brute_force_one_block_128cubed():
    rng = np.random.default_rng(21)
    a = random_codes((128, 128), rng)
    b = random_codes((128, 128), rng)
    sa = rng.uniform(1e-3, 2.0, size=(1, 128)).astype(np.float32)      # [K/128][M]
    sb = rng.uniform(1e-3, 2.0, size=(1, 1)).astype(np.float32)        # [N/128][K/128]
    acc, y, _ = oracle.gemm_fprop(a, sa, b, sb)
    P = block_partials(a, b)[:, :, 0]
    # One block: acc = fma(P, sa*sb, 0) = RN32(RN32(P) * RN32(sa*sb)); the
    # product of two FP32 values is exact in float64, so one float64->float32
    # rounding of it is the correctly rounded result.
    p32 = (P.astype(np.float64) / 2.0 ** 18).astype(np.float32)
    s = (sa[0][:, None] * sb[0, 0]).astype(np.float32)
    expect = (p32.astype(np.float64) * s.astype(np.float64)).astype(np.float32)
    assert np.array_equal(acc, expect)
    ref_bf16 = torch.from_numpy(expect).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y, ref_bf16)


def test_promotion_chain_bit_exact_multi_block():
    rng = np.random.default_rng(22)
    M, N, K = 6, 256, 640          # 5 K-blocks, 2 weight row-blocks
    a = random_codes((M, K), rng)
    b = random_codes((N, K), rng)
    sa = (rng.uniform(0.5, 1.5, size=(K // 128, M)) * 2.0 ** rng.integers(-20, 10, size=(K // 128, M))).astype(np.float32)
    sb = (rng.uniform(0.5, 1.5, size=(N // 128, K // 128)) * 2.0 ** rng.integers(-20, 10, size=(N // 128, K // 128))).astype(np.float32)
    acc, _, _ = oracle.gemm_fprop(a, sa, b, sb)
    P = block_partials(a, b)
    for m in range(M):
        for n in range(0, N, 7):
            e = emulate_promotion(P[m, n], sa[:, m], sb[n // 128, :])
            assert acc[m, n] == np.float32(e), (m, n)


def dequant_rows(codes, scales_per_block):
    """codes [r][k], scales [r][k/128] -> float64 dequantized values."""
    v = oracle.e4m3_decode(codes)
    return v * np.repeat(scales_per_block.astype(np.float64), 128, axis=1)


def test_fprop_against_float64_within_promotion_bound():
    x = inputs.random_bf16((128, 1024), seed=31)
    x[:, 5] *= 50.0
    w = inputs.random_bf16((384, 1024), seed=32, std=0.02)
    xq, sx = oracle.quant_rowwise_1x128(x)
    wq, _, sw = oracle.quant_weight_128x128(w)
    acc, _, sab = oracle.gemm_fprop(xq, sx, wq, sw)
    A = dequant_rows(xq, sx.T)
    B = dequant_rows(wq, np.repeat(sw, 128, axis=0))
    f64 = A @ B.T
    absprod = np.abs(A) @ np.abs(B).T
    assert np.allclose(sab, absprod, rtol=1e-12, atol=0)
    kb = 1024 // 128
    assert np.all(np.abs(acc.astype(np.float64) - f64) <= (kb + 2) * 2.0 ** -24 * absprod)


def test_unit_scales_reduce_to_integer_matmul():
    rng = np.random.default_rng(33)
    vals = np.arange(-16, 17, dtype=np.float32)
    codes_of = {float(v): int(oracle.e4m3_encode(np.array([v], np.float32))[0]) for v in vals}
    ai = rng.integers(-16, 17, size=(8, 256))
    bi = rng.integers(-16, 17, size=(128, 256))
    a = np.vectorize(lambda v: codes_of[float(v)])(ai).astype(np.uint8)
    b = np.vectorize(lambda v: codes_of[float(v)])(bi).astype(np.uint8)
    acc, _, _ = oracle.gemm_fprop(a, np.ones((2, 8), np.float32), b, np.ones((1, 2), np.float32))
    assert np.array_equal(acc.astype(np.int64), ai @ bi.T)


def test_dgrad_equals_fprop_on_transposed_weight():
    rng = np.random.default_rng(34)
    M, N, K = 8, 384, 256
    dy = random_codes((M, N), rng)
    w = random_codes((N, K), rng)
    sdy = rng.uniform(0.1, 2, size=(N // 128, M)).astype(np.float32)
    sw = rng.uniform(0.1, 2, size=(N // 128, K // 128)).astype(np.float32)
    acc_d, y_d, s_d = oracle.gemm_dgrad(dy, sdy, w, sw)
    # dX = dY W is fprop with B = W^T [K][N], whose 128x128 block scales are sw^T.
    acc_f, y_f, s_f = oracle.gemm_fprop(dy, sdy, np.ascontiguousarray(w.T), np.ascontiguousarray(sw.T))
    assert np.array_equal(acc_d, acc_f) and np.array_equal(y_d, y_f)
    # and against the float64 product within the bound
    A = dequant_rows(dy, sdy.T)
    Wd = oracle.e4m3_decode(w) * np.repeat(np.repeat(sw, 128, axis=0), 128, axis=1)
    f64 = A @ Wd
    absprod = np.abs(A) @ np.abs(Wd)
    assert np.all(np.abs(acc_d - f64) <= (N // 128 + 2) * 2.0 ** -24 * absprod)


def test_wgrad_against_float64_and_brute_force():
    rng = np.random.default_rng(35)
    M, N, K = 384, 128, 256        # tokens, out features, in features
    dyT = random_codes((N, M), rng)
    xT = random_codes((K, M), rng)
    sdyT = rng.uniform(0.1, 2, size=(M // 128, N)).astype(np.float32)
    sxT = rng.uniform(0.1, 2, size=(M // 128, K)).astype(np.float32)
    rows = np.array([0, 5, 77, 127])
    acc, _, _ = oracle.gemm_wgrad(dyT, sdyT, xT, sxT, rows=rows)
    P = block_partials(dyT, xT)                     # [N][K][blocks]
    for i, n in enumerate(rows):
        for k in range(0, K, 13):
            e = emulate_promotion(P[n, k], sdyT[:, n], sxT[:, k])
            assert acc[i, k] == np.float32(e)
    A = dequant_rows(dyT, sdyT.T)
    B = dequant_rows(xT, sxT.T)
    f64 = (A @ B.T)[rows]
    absprod = (np.abs(A) @ np.abs(B).T)[rows]
    assert np.all(np.abs(acc - f64) <= (M // 128 + 2) * 2.0 ** -24 * absprod)


def test_row_subset_matches_full():
    x = inputs.random_bf16((256, 256), seed=36)
    w = inputs.random_bf16((256, 256), seed=37, std=0.02)
    xq, sx = oracle.quant_rowwise_1x128(x)
    wq, _, sw = oracle.quant_weight_128x128(w)
    full, _, _ = oracle.gemm_fprop(xq, sx, wq, sw)
    rows = np.array([3, 100, 255])
    sub, _, _ = oracle.gemm_fprop(xq, sx, wq, sw, rows=rows)
    assert np.array_equal(sub, full[rows])
