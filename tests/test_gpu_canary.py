"""Canary bytes around every output buffer and around the split-K scratch.

Each entry point writes through TMA tensor maps and plain stores whose
extents the host derives from the call's sizes; a wrong extent, a stray
tile or a misplaced partial would write outside the caller's buffer.  Here
every output is a view into a larger allocation whose first and last
4 KiB hold a fixed pattern, on shapes with a token tail and a half-width
last output tile, and the pattern must survive each call."""
import numpy as np
import pytest
import torch

from fp8_block_scaled_16_b300 import binding as B
from fp8_block_scaled_16_b300 import inputs
from fp8_block_scaled_16_b300.linear import interleave_gate_up

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.load()
    yield
    torch.cuda.synchronize()


class Guarded:
    """A tensor of `shape`/`dtype` with GUARD pattern bytes on both sides."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        self.raw = torch.full((2 * GUARD + n,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(*shape)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        head, tail = self.raw[:GUARD], self.raw[GUARD + self.n:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def check(what, *bufs):
    assert B.fp8bs_get_device_status() == 0, what
    for i, g in enumerate(bufs):
        assert g.intact(), f"{what}: bytes outside output {i} were written"


M, N, K = 300, 640, 768        # token tail (Mp = 384); N = 2.5 tiles of 256 columns
MP = B.padded_tokens(M)


@pytest.fixture(scope="module")
def operands():
    x = inputs.random_bf16((M, K), seed=501)
    w = inputs.random_bf16((N, K), seed=502, std=0.02)
    dy = inputs.random_bf16((M, N), seed=503, std=1e-3)
    xq, sx, xTq, sxT = B.fp8bs_quantize_act(x.cuda(), B.ROWWISE | B.COLWISE_T)
    wq, wqT, sw = B.fp8bs_quantize_weight(w.cuda(), want_t=True)
    dyq, sdy, dyTq, sdyT = B.fp8bs_quantize_act(dy.cuda(), B.ROWWISE | B.COLWISE_T)
    return dict(x=x.cuda(), w=w.cuda(), xq=xq, sx=sx, xTq=xTq, sxT=sxT, wq=wq, wqT=wqT, sw=sw, dyq=dyq, sdy=sdy,
                dyTq=dyTq, sdyT=sdyT)


def test_quantizers_stay_in_their_outputs(operands):
    q, s = Guarded((M, K), torch.uint8), Guarded((K // 128, MP), torch.float32)
    qT, sT = Guarded((K, MP), torch.uint8), Guarded((MP // 128, K), torch.float32)
    B.fp8bs_quantize_act(operands["x"], B.ROWWISE | B.COLWISE_T, q=q.t, s=s.t, qT=qT.t, sT=sT.t)
    check("quantize_act", q, s, qT, sT)
    wq, wqT, sw = Guarded((N, K), torch.uint8), Guarded((K, N), torch.uint8), Guarded((N // 128, K // 128),
                                                                                       torch.float32)
    B.fp8bs_quantize_weight(operands["w"], q=wq.t, qT=wqT.t, s=sw.t)
    check("quantize_weight", wq, wqT, sw)
    assert torch.equal(q.t, operands["xq"]) and torch.equal(wqT.t, operands["wqT"])


def test_gemms_stay_in_their_outputs(operands):
    o = operands
    y = Guarded((M, N), torch.bfloat16)
    B.fp8bs_gemm_fprop(o["xq"], o["sx"], o["wq"], o["sw"], y=y.t)
    check("fprop", y)
    yq, sy = Guarded((M, N), torch.uint8), Guarded((N // 128, MP), torch.float32)
    y2 = Guarded((M, N), torch.bfloat16)
    B.fp8bs_gemm_fprop_quant(o["xq"], o["sx"], o["wq"], o["sw"], y=y2.t, yq=yq.t, sy=sy.t)
    check("fprop_quant", y2, yq, sy)
    assert torch.equal(y.t, y2.t)
    dx = Guarded((M, K), torch.bfloat16)
    B.fp8bs_gemm_dgrad(o["dyq"], o["sdy"], o["wqT"], o["sw"], dx=dx.t)
    check("dgrad", dx)
    dw = Guarded((N, K), torch.bfloat16)
    B.fp8bs_gemm_wgrad(o["dyTq"], o["sdyT"], o["xTq"], o["sxT"], dw=dw.t)
    check("wgrad", dw)
    acc = Guarded((N, K), torch.float32)
    acc.t.zero_()
    B.fp8bs_gemm_wgrad_accumulate_f32(o["dyTq"], o["sdyT"], o["xTq"], o["sxT"], acc.t)
    check("wgrad_accumulate_f32", acc)
    ys = [Guarded((M, N), torch.bfloat16), Guarded((M, K), torch.bfloat16)]
    B.fp8bs_gemm_group([(B.OP_FPROP, o["xq"], o["sx"], o["wq"], o["sw"], ys[0].t),
                        (B.OP_DGRAD, o["dyq"], o["sdy"], o["wqT"], o["sw"], ys[1].t)])
    check("group", *ys)
    assert torch.equal(ys[0].t, y.t) and torch.equal(ys[1].t, dx.t)


def test_swiglu_forward_stays_in_its_outputs():
    I = 384                                   # 3 H blocks; gate+up weight of 2I rows
    x = inputs.random_bf16((M, K), seed=511)
    wg = inputs.random_bf16((I, K), seed=512, std=0.02)
    wu = inputs.random_bf16((I, K), seed=513, std=0.02)
    xq, sx, _, _ = B.fp8bs_quantize_act(x.cuda(), B.ROWWISE)
    wq, _, sw = B.fp8bs_quantize_weight(interleave_gate_up(wg, wu).cuda(), want_t=False)
    h, hq, sh = Guarded((M, I), torch.bfloat16), Guarded((M, I), torch.uint8), Guarded((I // 128, MP),
                                                                                       torch.float32)
    B.fp8bs_gemm_fprop_swiglu_quant(xq, sx, wq, sw, h=h.t, hq=hq.t, sh=sh.t)
    check("fprop_swiglu_quant", h, hq, sh)


def test_split_k_stays_in_its_scratch():
    """A weight gradient whose plan splits every tile, with the registered
    scratch itself guarded: partials and arrival counters stay inside it."""
    Ms, Ns, Ks = 8192, 256, 512
    need = B.fp8bs_gemm_wgrad_workspace_bytes(Ms, Ns, Ks)
    assert need > 0, "this shape should split"
    x = inputs.random_bf16((Ms, Ks), seed=521)
    dy = inputs.random_bf16((Ms, Ns), seed=522, std=1e-3)
    _, _, xTq, sxT = B.fp8bs_quantize_act(x.cuda(), B.COLWISE_T)
    _, _, dyTq, sdyT = B.fp8bs_quantize_act(dy.cuda(), B.COLWISE_T)
    ws = Guarded((need,), torch.uint8)
    torch.cuda.synchronize()
    B.fp8bs_set_workspace(ws.t)
    try:
        dw = Guarded((Ns, Ks), torch.bfloat16)
        B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT, dw=dw.t)
        check("split wgrad", dw, ws)
        ref = B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT, split=False)
        assert B.fp8bs_get_device_status() == 0
        assert (dw.t.float() - ref.float()).abs().max().item() <= 2.0 ** -6 * ref.float().abs().max().item()
    finally:
        torch.cuda.synchronize()
        B.fp8bs_set_workspace(None)
