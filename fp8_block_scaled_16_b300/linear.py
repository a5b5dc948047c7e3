"""One FP8 block-scaled linear layer, forward and backward, as a fixed
sequence of library calls on preallocated device buffers.

    forward : X -> (Xq, sX) [1x128] and (XTq, sXT) [128x1, transposed] in one
              read of X; W -> (Wq, WqT, sW) [128x128]; Y = X W^T
    backward: dY -> (dYq, sdY) and (dYTq, sdYT) in one read of dY;
              dX = dY W; dW = dY^T X

This is the linear-layer GEMM path the Puro-2B pages put on blockwise FP8
(blog section "FP8：加快 RTX 5090 上的训练"; arXiv part 1/7, section 2.1):
the main GEMMs of forward and backward, with activations requantized along
tokens for the weight gradient.  The weight is quantized inside every step
here; a trainer that keeps W fixed across micro-batches may quantize it once.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List

import torch

from . import binding as B


@dataclass
class Launch:
    op: str        # "quant_act", "quant_weight", "fprop", "dgrad", "wgrad"
    work: int      # algorithmic FLOPs (GEMMs) or bytes (quantizers)
    unit: str      # "flops" or "bytes"
    run: Callable[[], object]


class Fp8LinearStep:
    """Buffers for one linear of shape x [M][K], w [N][K] and the calls of
    one training step over them."""

    def __init__(self, M: int, N: int, K: int, device="cuda", ops=("fprop", "dgrad", "wgrad")):
        self.M, self.N, self.K, self.ops = M, N, K, tuple(ops)
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=device)  # noqa: E731
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        need_t = "wgrad" in self.ops
        Mp = B.padded_tokens(M)  # token-major arrays: tokens rounded up to 128
        self.xq, self.sx = e((M, K), u8), e((K // 128, Mp), f32)
        self.xTq, self.sxT = (e((K, Mp), u8), e((Mp // 128, K), f32)) if need_t else (None, None)
        self.wq, self.sw = e((N, K), u8), e((N // 128, K // 128), f32)
        self.wqT = e((K, N), u8) if "dgrad" in self.ops else None
        self.y = e((M, N), bf)
        bwd = "dgrad" in self.ops or "wgrad" in self.ops
        self.dyq, self.sdy = (e((M, N), u8), e((N // 128, Mp), f32)) if "dgrad" in self.ops else (None, None)
        self.dyTq, self.sdyT = (e((N, Mp), u8), e((Mp // 128, N), f32)) if need_t else (None, None)
        self.dx = e((M, K), bf) if "dgrad" in self.ops else None
        self.dw = e((N, K), bf) if "wgrad" in self.ops else None
        self.has_bwd = bwd

    def launch_list(self, x, w, dy=None, stream=None) -> List[Launch]:
        """The step's library calls in order, each with its algorithmic work:
        FLOPs (2 M N K) for a GEMM, bytes moved for a quantizer (BF16 read,
        E4M3 written per requested layout, 4 bytes per scale)."""
        M, N, K = self.M, self.N, self.K
        wgrad, dgrad = "wgrad" in self.ops, "dgrad" in self.ops
        xflags = B.ROWWISE | (B.COLWISE_T if wgrad else 0)
        dyflags = (B.ROWWISE if dgrad else 0) | (B.COLWISE_T if wgrad else 0)

        def act_bytes(rows, cols, flags):
            n = rows * cols
            layouts = bin(flags).count("1")
            return 2 * n + layouts * (n + 4 * n // 128)

        out = [
            Launch("quant_act", act_bytes(M, K, xflags), "bytes",
                   lambda: B.fp8bs_quantize_act(x, xflags, self.xq, self.sx, self.xTq, self.sxT, stream=stream)),
            Launch("quant_weight", 2 * N * K + N * K * (2 if dgrad else 1) + 4 * (N // 128) * (K // 128), "bytes",
                   lambda: B.fp8bs_quantize_weight(w, self.wq, self.wqT, self.sw, want_t=dgrad, stream=stream)),
            Launch("fprop", 2 * M * N * K, "flops",
                   lambda: B.fp8bs_gemm_fprop(self.xq, self.sx, self.wq, self.sw, self.y, stream=stream)),
        ]
        if self.has_bwd:
            out.append(Launch("quant_act", act_bytes(M, N, dyflags), "bytes",
                              lambda: B.fp8bs_quantize_act(dy, dyflags, self.dyq, self.sdy, self.dyTq, self.sdyT,
                                                           stream=stream)))
        if dgrad:
            out.append(Launch("dgrad", 2 * M * N * K, "flops",
                              lambda: B.fp8bs_gemm_dgrad(self.dyq, self.sdy, self.wqT, self.sw, self.dx,
                                                         stream=stream)))
        if wgrad:
            out.append(Launch("wgrad", 2 * M * N * K, "flops",
                              lambda: B.fp8bs_gemm_wgrad(self.dyTq, self.sdyT, self.xTq, self.sxT, self.dw,
                                                         stream=stream)))
        return out

    def step(self, x, w, dy=None, stream=None):
        for launch in self.launch_list(x, w, dy, stream=stream):
            launch.run()
        return self.y, self.dx, self.dw


def grouped_launch_list(steps, stream=None) -> List[Launch]:
    """One training step of several independent linears (e.g. a decoder
    layer's four) with each GEMM phase in one grouped launch.  `steps` lists
    (Fp8LinearStep, x, w, dy): the quantizations run per linear as in
    launch_list; then one launch computes every forward product, one every
    data gradient and one every weight gradient (fp8bs_gemm_group).  The
    outputs are bitwise those of the linears' own launch lists without
    split-K."""
    if len(steps) > B.GROUP_MAX:
        raise ValueError(f"at most {B.GROUP_MAX} linears per group")
    quant_x, quant_dy, fprop, dgrad, wgrad = [], [], [], [], []
    for st, x, w, dy in steps:
        single = st.launch_list(x, w, dy, stream=stream)
        quant_x += [l for l in single if l.op == "quant_weight" or (l.op == "quant_act" and l is single[0])]
        quant_dy += [l for l in single if l.op == "quant_act" and l is not single[0]]
        fl = 2 * st.M * st.N * st.K
        fprop.append(((B.OP_FPROP, st.xq, st.sx, st.wq, st.sw, st.y), fl))
        if "dgrad" in st.ops:
            dgrad.append(((B.OP_DGRAD, st.dyq, st.sdy, st.wqT, st.sw, st.dx), fl))
        if "wgrad" in st.ops:
            wgrad.append(((B.OP_WGRAD, st.dyTq, st.sdyT, st.xTq, st.sxT, st.dw), fl))

    def group(op, members):
        args = [m for m, _ in members]
        return Launch(op, sum(f for _, f in members), "flops", lambda: B.fp8bs_gemm_group(args, stream=stream))

    out = quant_x + [group("fprop", fprop)] + quant_dy
    if dgrad:
        out.append(group("dgrad", dgrad))
    if wgrad:
        out.append(group("wgrad", wgrad))
    return out


def interleave_gate_up(w_gate: torch.Tensor, w_up: torch.Tensor) -> torch.Tensor:
    """The gate+up weight in the row order fp8bs_gemm_fprop_swiglu_quant
    reads: 128-row blocks alternating gate block j, up block j ([2I][K] from
    two [I][K] weights, I a multiple of 128).  A weight layout chosen once,
    when the weights are loaded."""
    I, K = w_gate.shape
    if tuple(w_up.shape) != (I, K) or I % 128:
        raise ValueError("gate and up weights must both be [I][K] with I a multiple of 128")
    return torch.stack([w_gate.reshape(I // 128, 128, K), w_up.reshape(I // 128, 128, K)], 1).reshape(2 * I, K)


class Fp8LinearFunction(torch.autograd.Function):
    """y = x W^T through the FP8 block-scaled path, as a torch autograd op.

    forward : X -> 1x128 (and, if W needs a gradient, 128x1 transposed) in one
              read; W -> 128x128 blocks (and W^T if X needs a gradient);
              Y = fp8bs_gemm_fprop.
    backward: dY -> 1x128 (for dX) and/or 128x1 transposed (for dW) in one
              read; dX = fp8bs_gemm_dgrad, dW = fp8bs_gemm_wgrad.

    x: BF16 CUDA tensor [..., K]; w: BF16 [N][K]; K and N multiples of 128,
    any number of tokens.  Only the quantized operands the backward needs are
    kept (Xq^T and its scales, Wq^T and the block scales): 1 byte per element
    instead of the BF16 originals.  Every arithmetic step runs in the
    library's kernels; this class only orders the calls."""

    @staticmethod
    def forward(ctx, x, w):
        K = x.shape[-1]
        N = w.shape[0]
        if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16 or not x.is_cuda:
            raise TypeError("Fp8LinearFunction takes BF16 CUDA tensors")
        if tuple(w.shape) != (N, K) or K % 128 or N % 128:
            raise ValueError("w must be [N][K] with N and K multiples of 128, x [..., K]")
        x2 = x.reshape(-1, K).contiguous()
        need_dw, need_dx = ctx.needs_input_grad[1], ctx.needs_input_grad[0]
        xq, sx, xTq, sxT = B.fp8bs_quantize_act(x2, B.ROWWISE | (B.COLWISE_T if need_dw else 0))
        wq, wqT, sw = B.fp8bs_quantize_weight(w.contiguous(), want_t=need_dx)
        y = B.fp8bs_gemm_fprop(xq, sx, wq, sw)
        ctx.save_for_backward(xTq, sxT, wqT, sw)
        ctx.x_shape, ctx.M, ctx.N, ctx.K = x.shape, x2.shape[0], N, K
        return y.reshape(*x.shape[:-1], N)

    @staticmethod
    def backward(ctx, dy):
        xTq, sxT, wqT, sw = ctx.saved_tensors
        need_dx, need_dw = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        dy2 = dy.reshape(-1, ctx.N)
        if dy2.dtype != torch.bfloat16:
            dy2 = dy2.to(torch.bfloat16)
        dy2 = dy2.contiguous()
        flags = (B.ROWWISE if need_dx else 0) | (B.COLWISE_T if need_dw else 0)
        dyq, sdy, dyTq, sdyT = B.fp8bs_quantize_act(dy2, flags)
        dx = B.fp8bs_gemm_dgrad(dyq, sdy, wqT, sw).reshape(ctx.x_shape) if need_dx else None
        dw = B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT) if need_dw else None
        return dx, dw


class Fp8Linear(torch.nn.Module):
    """A bias-free linear layer whose forward and backward GEMMs run on the
    FP8 block-scaled path (the weight is kept in BF16 and quantized in every
    forward)."""

    def __init__(self, in_features: int, out_features: int, device="cuda", std: float = 0.02):
        super().__init__()
        if in_features % 128 or out_features % 128:
            raise ValueError("in_features and out_features must be multiples of 128")
        self.in_features, self.out_features = in_features, out_features
        self.weight = torch.nn.Parameter(
            torch.randn(out_features, in_features, device=device, dtype=torch.float32).mul_(std).to(torch.bfloat16))

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return Fp8LinearFunction.apply(x, self.weight)
