"""GPU parity of the SwiGLU forward (gate+up projection with SiLU(g) * u and
the down projection's FP8 input in the GEMM epilogue), through the C ABI.

1. The activation itself (fp8bs_debug_silu_mul) equals the oracle's bit for
   bit on every finite BF16 gate value in [-100, 100] and on seeded pairs.
2. The fused product's BF16 H equals the activation applied to the plain
   forward product's gate and up outputs (bitwise), its E4M3 payload and
   scales equal the row-wise quantizer's on that H (bitwise), and H stays
   within the oracle's GEMM tolerance carried through the activation."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_16_b300 import binding as B
from fp8_block_scaled_16_b300 import inputs
from fp8_block_scaled_16_b300.linear import interleave_gate_up
from tests._parity import np_bf16_bits, oracle_gemm_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.load()
    yield
    torch.cuda.synchronize()


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_bf16_cuda(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def test_activation_matches_oracle_bit_for_bit():
    all_bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = bf16_to_f64(all_bits)
    g = all_bits[np.isfinite(v) & (np.abs(v) <= 100.0)]
    cases = []
    for uval in (1.0, -0.75, 3.5, 1e-3, -250.0):
        ub = np.float32(uval).view(np.uint32) >> 16
        cases.append((g, np.full(g.shape, ub, np.uint16)))
    gr = np_bf16_bits(inputs.random_bf16((1 << 20,), seed=901, std=3.0))
    ur = np_bf16_bits(inputs.random_bf16((1 << 20,), seed=902, std=1.0))
    cases.append((gr, ur))
    for gb, ub in cases:
        h = B.fp8bs_debug_silu_mul(to_bf16_cuda(gb), to_bf16_cuda(ub))
        assert B.fp8bs_get_device_status() == 0
        assert np.array_equal(np_bf16_bits(h), oracle.silu_mul(gb, ub))


def split_gate_up(a: np.ndarray, I: int):
    """[rows][2I] in the interleaved column order -> (gate, up), each [rows][I]."""
    r = a.reshape(a.shape[0], I // 128, 2, 128)
    return r[:, :, 0, :].reshape(-1, I), r[:, :, 1, :].reshape(-1, I)


@pytest.mark.parametrize("M,I,K", [
    (300, 384, 640),      # token tail; 3 H blocks
    (2048, 1408, 2048),   # 16 x 11 tiles of the interleaved gate+up weight
])
def test_fused_swiglu_forward(M, I, K):
    x = inputs.random_bf16((M, K), seed=70 + M)
    wg = inputs.random_bf16((I, K), seed=71 + I, std=0.02)
    wu = inputs.random_bf16((I, K), seed=72 + I, std=0.02)
    w = interleave_gate_up(wg, wu)
    xq, sx, _, _ = B.fp8bs_quantize_act(x.cuda(), B.ROWWISE)
    wq, _, sw = B.fp8bs_quantize_weight(w.cuda(), want_t=False)
    h, hq, sh = B.fp8bs_gemm_fprop_swiglu_quant(xq, sx, wq, sw)
    _, hq2, sh2 = B.fp8bs_gemm_fprop_swiglu_quant(xq, sx, wq, sw, want_bf16=False)
    y = B.fp8bs_gemm_fprop(xq, sx, wq, sw)                         # interleaved [M][2I]
    assert B.fp8bs_get_device_status() == 0
    yb = y.view(M, I // 128, 2, 128)
    h_ref = B.fp8bs_debug_silu_mul(yb[:, :, 0, :].reshape(M, I).contiguous(),
                                   yb[:, :, 1, :].reshape(M, I).contiguous())
    assert torch.equal(h.view(torch.int16), h_ref.view(torch.int16))
    q_ref, s_ref, _, _ = B.fp8bs_quantize_act(h, B.ROWWISE)
    assert torch.equal(hq, q_ref) and torch.equal(sh.view(torch.int32), s_ref.view(torch.int32))
    assert torch.equal(hq2, hq) and torch.equal(sh2.view(torch.int32), sh.view(torch.int32))

    # Against the oracle: its product of the same quantized operands, through
    # its activation; the GEMM tolerance carried through SiLU(g) * u
    # (|SiLU'| <= 1.1, |SiLU(g)| <= |g|) plus both sides' BF16 roundings.
    rows = np.arange(M) if M <= 512 else inputs.sample_rows(M, 7070, 64).numpy()
    oxq, osx = oracle.quant_rowwise_1x128(x)
    owq, _, osw = oracle.quant_weight_128x128(w, want_t=False)
    acc, bits, sab = oracle_gemm_rows("fprop", oxq, osx, owq, osw, rows)
    g_acc, u_acc = split_gate_up(acc.astype(np.float64), I)
    g_bits, u_bits = split_gate_up(bits, I)
    g_sab, u_sab = split_gate_up(sab, I)
    h_ora = bf16_to_f64(oracle.silu_mul(g_bits, u_bits))
    g, u = bf16_to_f64(g_bits), bf16_to_f64(u_bits)
    eg = 2.0 ** -8 * np.abs(g_acc) + 1e-6 * g_sab + 2.0 ** -8 * np.abs(g)
    eu = 2.0 ** -8 * np.abs(u_acc) + 1e-6 * u_sab + 2.0 ** -8 * np.abs(u)
    bound = 1.1 * eg * np.abs(u) + np.abs(g) * eu + 1.1 * eg * eu + 2.0 ** -7 * np.abs(h_ora) + 1e-30
    got = bf16_to_f64(np_bf16_bits(h)[rows])
    assert np.all(np.abs(got - h_ora) <= bound), float(np.max(np.abs(got - h_ora) - bound))
