"""The GEMMs' FP32 promotion accumulators against the oracle's, through the
FP32-output test mode (fp8bs_debug_set_flags(FP8BS_DEBUG_F32_OUT)): with no
BF16 rounding of the output, the comparison sees only the tensor core's
summation inside each 128-wide block and the promotion chain.

Bound (derived, not fitted).  The oracle sums each block exactly (double)
and rounds the sum once to FP32; the tensor core accumulates a block over
four K = 32 MMA steps in FP32.  With at most one FP32 rounding per step, of
a partial sum no larger than the block's sum of |a_k b_k|, a block's
partial differs by at most 5 * 2^-24 * sum_{k in b} |a_k b_k| (four step
roundings and the oracle's one); scaled by the block's scale and summed over
blocks: 5 * 2^-24 * sum_k |a_k b_k| over the dequantized operands.  Both
sides then run the same fmaf chain with the same FP32 scale products; a
difference in an input of one fma moves its result by that difference plus
at most one rounding (2^-24 of the running value, itself bounded by
sum |ab| up to rounding), which adds nb * 2^-24 * sum|ab| over nb blocks.
A K split into S parts adds S - 1 FP32 additions of partials (<= 4 more).
Rule:  |gpu - ref| <= (9 + nb) * 2^-24 * 1.01 * sum_k |a_k b_k|.
For comparison, the acceptance rule of the BF16 outputs allows
2^-8 |ref| + 1e-6 sum|ab|."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_16_b300 import binding as B
from fp8_block_scaled_16_b300 import inputs
from tests._parity import np_f32, oracle_gemm_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _f32_mode():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.load()
    B.fp8bs_debug_set_flags(B.DEBUG_F32_OUT)
    yield
    B.fp8bs_debug_set_flags(0)
    torch.cuda.synchronize()


def assert_f32_close(gpu: torch.Tensor, acc: np.ndarray, sab: np.ndarray, nb: int, what: str) -> float:
    g = np_f32(gpu).astype(np.float64)
    r = acc.astype(np.float64)
    tol = (9 + nb) * 2.0 ** -24 * 1.01 * sab
    err = np.abs(g - r)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} FP32 outputs outside (9 + {nb}) 2^-24 sum|ab|; "
                           f"first at {tuple(np.argwhere(bad)[0])}")
    return float((err / np.maximum(sab, 1e-300)).max())


def quantized_operands(M, N, K, seed):
    x = inputs.random_bf16((M, K), seed=seed)
    x[:, K // 5] *= 30.0
    w = inputs.random_bf16((N, K), seed=seed + 1, std=0.02)
    dy = inputs.random_bf16((M, N), seed=seed + 2, std=1e-3)
    return x, w, dy


@pytest.mark.parametrize("M,N,K", [
    (600, 1280, 1536),   # token tail, several tiles, 12 K blocks
    (128, 256, 4096),    # one tile, 32 K blocks
])
def test_forward_and_data_gradient_accumulators(M, N, K):
    x, w, dy = quantized_operands(M, N, K, seed=M + N + K)
    xq, sx, _, _ = B.fp8bs_quantize_act(x.cuda(), B.ROWWISE)
    wq, wqT, sw = B.fp8bs_quantize_weight(w.cuda(), want_t=True)
    dyq, sdy, _, _ = B.fp8bs_quantize_act(dy.cuda(), B.ROWWISE)
    y = B.fp8bs_gemm_fprop(xq, sx, wq, sw)
    dx = B.fp8bs_gemm_dgrad(dyq, sdy, wqT, sw)
    assert y.dtype == torch.float32 and dx.dtype == torch.float32
    assert B.fp8bs_get_device_status() == 0
    # The oracle on its own quantization of the same inputs (the quantizers'
    # bytes are checked bit for bit elsewhere).
    oxq, osx = oracle.quant_rowwise_1x128(x)
    owq, _, osw = oracle.quant_weight_128x128(w, want_t=False)
    odyq, osdy = oracle.quant_rowwise_1x128(dy)
    rows = np.arange(M)
    acc, _, sab = oracle_gemm_rows("fprop", oxq, osx, owq, osw, rows)
    worst_f = assert_f32_close(y, acc, sab, K // 128, "fprop")
    acc, _, sab = oracle_gemm_rows("dgrad", odyq, osdy, owq, osw, rows)
    worst_d = assert_f32_close(dx, acc, sab, N // 128, "dgrad")
    print(f"largest |gpu - ref| / sum|ab|: fprop {worst_f:.3g}, dgrad {worst_d:.3g}")


@pytest.mark.parametrize("M,N,K", [
    (1000, 512, 768),    # token tail in the contraction, unsplit
    (8192, 256, 512),    # 4 tiles, 64 K blocks: split across CTAs
])
def test_weight_gradient_accumulators(M, N, K):
    x, w, dy = quantized_operands(M, N, K, seed=3 * M + N + K)
    _, _, xTq, sxT = B.fp8bs_quantize_act(x.cuda(), B.COLWISE_T)
    _, _, dyTq, sdyT = B.fp8bs_quantize_act(dy.cuda(), B.COLWISE_T)
    dw = B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT)
    assert dw.dtype == torch.float32 and B.fp8bs_get_device_status() == 0
    oxTq, osxT = oracle.quant_colwise_128x1_T(x)
    odyTq, osdyT = oracle.quant_colwise_128x1_T(dy)
    acc, _, sab = oracle_gemm_rows("wgrad", odyTq, osdyT, oxTq, osxT, np.arange(N))
    worst = assert_f32_close(dw, acc, sab, B.padded_tokens(M) // 128, "wgrad")
    print(f"largest |gpu - ref| / sum|ab|: wgrad {worst:.3g}")


def test_mode_off_restores_bf16_outputs():
    B.fp8bs_debug_set_flags(0)
    x, w, _ = quantized_operands(256, 256, 256, seed=77)
    xq, sx, _, _ = B.fp8bs_quantize_act(x.cuda(), B.ROWWISE)
    wq, _, sw = B.fp8bs_quantize_weight(w.cuda(), want_t=False)
    assert B.fp8bs_gemm_fprop(xq, sx, wq, sw).dtype == torch.bfloat16
