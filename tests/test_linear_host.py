"""Host logic of the layer-step wrappers (no GPU): the order of a linear's
library calls, the algorithmic work each is charged with (the figures the
benchmark divides by), and the grouped step's structure.  Buffers live on the
CPU here; no call is run."""
import pytest

from fp8_block_scaled_16_b300 import binding as B
import torch

from fp8_block_scaled_16_b300.linear import Fp8LinearStep, grouped_launch_list, interleave_gate_up


def act_bytes(rows, cols, layouts):
    n = rows * cols
    return 2 * n + layouts * (n + 4 * n // 128)


def test_single_linear_calls_and_work():
    M, N, K = 300, 384, 640
    st = Fp8LinearStep(M, N, K, device="cpu")
    ll = st.launch_list(None, None, None)
    assert [l.op for l in ll] == ["quant_act", "quant_weight", "fprop", "quant_act", "dgrad", "wgrad"]
    assert [l.unit for l in ll] == ["bytes", "bytes", "flops", "bytes", "flops", "flops"]
    assert ll[0].work == act_bytes(M, K, 2)                       # X read once, both layouts written
    assert ll[1].work == 2 * N * K + 2 * N * K + 4 * (N // 128) * (K // 128)   # W, Wq and WqT, scales
    assert ll[3].work == act_bytes(M, N, 2)
    assert ll[2].work == ll[4].work == ll[5].work == 2 * M * N * K
    # token-major buffers use the padded token count
    Mp = B.padded_tokens(M)
    assert tuple(st.sx.shape) == (K // 128, Mp) and tuple(st.xTq.shape) == (K, Mp)
    assert tuple(st.sdyT.shape) == (Mp // 128, N) and tuple(st.dyTq.shape) == (N, Mp)


def test_forward_only_linear():
    st = Fp8LinearStep(256, 512, 512, device="cpu", ops=("fprop",))
    ll = st.launch_list(None, None)
    assert [l.op for l in ll] == ["quant_act", "quant_weight", "fprop"]
    assert ll[0].work == act_bytes(256, 512, 1)                   # row-wise layout only
    assert ll[1].work == 2 * 512 * 512 + 512 * 512 + 4 * 4 * 4    # no transposed weight copy
    assert st.xTq is None and st.wqT is None and st.dw is None


def test_grouped_step_structure():
    shapes = [(256, 384, 256), (256, 256, 256), (256, 1408, 256), (256, 256, 768)]   # the layer at 1/8 width
    steps = [(Fp8LinearStep(M, N, K, device="cpu"), None, None, None) for M, N, K in shapes]
    gl = grouped_launch_list(steps)
    ops = [l.op for l in gl]
    # quantize X and W per linear, one forward group, dY per linear, one data-gradient and one weight-gradient group
    assert ops == ["quant_act", "quant_weight"] * 4 + ["fprop"] + ["quant_act"] * 4 + ["dgrad", "wgrad"]
    flops = sum(2 * M * N * K for M, N, K in shapes)
    assert [l.work for l in gl if l.unit == "flops"] == [flops] * 3
    per_linear = [l for st, *_ in steps for l in st.launch_list(None, None, None)]
    assert sum(l.work for l in gl) == sum(l.work for l in per_linear)   # same work, 15 launches instead of 24
    assert len(gl) == 15 and len(per_linear) == 24


def test_grouped_step_rejects_more_linears_than_a_group_holds():
    steps = [(Fp8LinearStep(128, 256, 128, device="cpu"), None, None, None)] * (B.GROUP_MAX + 1)
    with pytest.raises(ValueError):
        grouped_launch_list(steps)


def test_interleave_gate_up_row_order():
    I, K = 384, 8
    wg = torch.arange(I * K, dtype=torch.float32).reshape(I, K)
    wu = -wg - 1
    w = interleave_gate_up(wg, wu)
    assert tuple(w.shape) == (2 * I, K)
    for j in range(I // 128):
        assert torch.equal(w[256 * j:256 * j + 128], wg[128 * j:128 * j + 128])
        assert torch.equal(w[256 * j + 128:256 * j + 256], wu[128 * j:128 * j + 128])
    with pytest.raises(ValueError):
        interleave_gate_up(wg[:100], wu[:100])


def test_autograd_wrapper_checks_its_arguments():
    from fp8_block_scaled_16_b300.linear import Fp8Linear, Fp8LinearFunction
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    w = torch.zeros(128, 256, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        Fp8LinearFunction.apply(x, w)              # CPU tensors: the path is CUDA only
    with pytest.raises(TypeError):
        Fp8LinearFunction.apply(x.float(), w)      # not BF16
    with pytest.raises(ValueError):
        Fp8Linear(200, 128, device="cpu")          # not a multiple of 128
