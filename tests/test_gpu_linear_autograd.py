"""The torch autograd form of the linear layer (Fp8LinearFunction /
Fp8Linear): its output and gradients are bitwise those of the library calls
it orders (themselves checked against the oracle elsewhere), for a token
count with a tail, a batch dimension, and each combination of inputs that
need a gradient; and they agree with a float64 matmul of the BF16 operands
to within the FP8 scheme's error."""
import pytest
import torch

from fp8_block_scaled_16_b300 import binding as B
from fp8_block_scaled_16_b300 import inputs
from fp8_block_scaled_16_b300.linear import Fp8Linear, Fp8LinearFunction

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.load()
    yield
    torch.cuda.synchronize()


def direct(x2, w, dy2):
    xq, sx, xTq, sxT = B.fp8bs_quantize_act(x2, B.ROWWISE | B.COLWISE_T)
    wq, wqT, sw = B.fp8bs_quantize_weight(w, want_t=True)
    y = B.fp8bs_gemm_fprop(xq, sx, wq, sw)
    dyq, sdy, dyTq, sdyT = B.fp8bs_quantize_act(dy2, B.ROWWISE | B.COLWISE_T)
    return y, B.fp8bs_gemm_dgrad(dyq, sdy, wqT, sw), B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT)


def bits(t):
    return t.contiguous().view(torch.int16)


@pytest.mark.parametrize("grads", [(True, True), (True, False), (False, True)])
def test_autograd_matches_the_library_calls(grads):
    Bt, T, K, N = 2, 150, 640, 384       # 300 tokens: a tail of 44 in the last 128-token block
    x = inputs.random_bf16((Bt, T, K), seed=601).cuda()
    w = inputs.random_bf16((N, K), seed=602, std=0.02).cuda()
    dy = inputs.random_bf16((Bt, T, N), seed=603, std=1e-3).cuda()
    xa = x.clone().requires_grad_(grads[0])
    wa = w.clone().requires_grad_(grads[1])
    y = Fp8LinearFunction.apply(xa, wa)
    y.backward(dy)
    assert B.fp8bs_get_device_status() == 0
    y_ref, dx_ref, dw_ref = direct(x.reshape(-1, K), w, dy.reshape(-1, N))
    assert y.shape == (Bt, T, N) and torch.equal(bits(y.reshape(-1, N)), bits(y_ref))
    if grads[0]:
        assert xa.grad.shape == x.shape and torch.equal(bits(xa.grad.reshape(-1, K)), bits(dx_ref))
    else:
        assert xa.grad is None
    if grads[1]:
        assert torch.equal(bits(wa.grad), bits(dw_ref))
    else:
        assert wa.grad is None


def test_module_against_float64_reference():
    torch.manual_seed(0)
    M, K, N = 512, 1024, 768
    lin = Fp8Linear(K, N)
    x = inputs.random_bf16((M, K), seed=611).cuda().requires_grad_(True)
    dy = inputs.random_bf16((M, N), seed=612, std=1e-3).cuda()
    y = lin(x)
    y.backward(dy)
    assert B.fp8bs_get_device_status() == 0
    xd, wd, dyd = x.detach().double(), lin.weight.detach().double(), dy.double()
    for got, ref in ((y, xd @ wd.T), (x.grad, dyd @ wd), (lin.weight.grad, dyd.T @ xd)):
        err = (got.double() - ref).norm() / ref.norm()
        assert err < 0.05, float(err)   # E4M3 operands: ~2^-4 relative per element, averaging down
