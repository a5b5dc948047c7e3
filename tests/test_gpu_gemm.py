"""GPU parity of the block-scaled GEMMs against the oracle, through the C ABI.

Each case runs one linear layer's step on the GPU (quantize X, W, dY; fprop,
dgrad, wgrad), checks every quantized operand bit-exactly against the
oracle's, then checks the GEMM outputs against the oracle's unrounded FP32
accumulators with the acceptance rule in tests/_parity.py: on every output
for the small cases, and on 256 seeded random rows (randperm under seed + 1000)
for the full-size workloads."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_16_b300 import binding as B
from fp8_block_scaled_16_b300 import inputs
from fp8_block_scaled_16_b300.linear import Fp8LinearStep
from tests._parity import assert_gemm_close, np_bf16_bits, np_f32, np_u8, oracle_gemm_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.load()
    yield
    torch.cuda.synchronize()


def same_bits(gpu: torch.Tensor, ref: np.ndarray, what: str):
    g = np_u8(gpu) if gpu.dtype == torch.uint8 else np_f32(gpu).view(np.uint32)
    r = ref if ref.dtype == np.uint8 else ref.view(np.uint32)
    assert np.array_equal(g, r), f"{what} differs from the oracle"


def check_linear(x, w, dy, ops, seed, sample=None):
    """Run one linear's step on the GPU and compare everything with the
    oracle.  sample=None checks every output row."""
    M, K = x.shape
    N = w.shape[0]
    st = Fp8LinearStep(M, N, K, ops=ops)
    y, dx, dw = st.step(x.cuda(), w.cuda(), dy.cuda() if dy is not None else None)
    assert B.fp8bs_get_device_status() == 0
    torch.cuda.synchronize()

    oxq, osx = oracle.quant_rowwise_1x128(x)
    owq, owqT, osw = oracle.quant_weight_128x128(w, want_t="dgrad" in ops)
    same_bits(st.xq, oxq, "Xq")
    same_bits(st.sx, osx, "sX")
    same_bits(st.wq, owq, "Wq")
    same_bits(st.sw, osw, "sW")

    def rows_of(total):
        if sample is None:
            return np.arange(total)
        return inputs.sample_rows(total, seed + 1000, sample).numpy()

    worst = {}
    r = rows_of(M)
    acc, _, sab = oracle_gemm_rows("fprop", oxq, osx, owq, osw, r)
    worst["fprop"] = assert_gemm_close(np_bf16_bits(y)[r], acc, sab, "fprop")
    if "dgrad" in ops:
        same_bits(st.wqT, owqT, "WqT")
        odyq, osdy = oracle.quant_rowwise_1x128(dy)
        same_bits(st.dyq, odyq, "dYq")
        same_bits(st.sdy, osdy, "sdY")
        acc, _, sab = oracle_gemm_rows("dgrad", odyq, osdy, owq, osw, r)
        worst["dgrad"] = assert_gemm_close(np_bf16_bits(dx)[r], acc, sab, "dgrad")
    if "wgrad" in ops:
        oxTq, osxT = oracle.quant_colwise_128x1_T(x)
        odyTq, osdyT = oracle.quant_colwise_128x1_T(dy)
        same_bits(st.xTq, oxTq, "XTq")
        same_bits(st.sxT, osxT, "sXT")
        same_bits(st.dyTq, odyTq, "dYTq")
        same_bits(st.sdyT, osdyT, "sdYT")
        rn = rows_of(N)
        acc, _, sab = oracle_gemm_rows("wgrad", odyTq, osdyT, oxTq, osxT, rn)
        worst["wgrad"] = assert_gemm_close(np_bf16_bits(dw)[rn], acc, sab, "wgrad")
    return worst


@pytest.mark.parametrize("M,N,K", [
    (128, 128, 128),      # one tile, one K block, N below the tile width
    (384, 384, 640),      # ragged N tile (384 = 256 + 128), 5 K blocks
    (256, 640, 384),      # dgrad output 384 wide: ragged; wgrad contracts 256 tokens
    (1152, 1280, 1024),   # more tiles than a fraction of the SMs, several per CTA
])
def test_small_shapes_full_outputs(M, N, K):
    seed = M * 7 + N * 3 + K
    x = inputs.random_bf16((M, K), seed=seed)
    x[:, K // 3] *= 40.0
    w = inputs.random_bf16((N, K), seed=seed + 1, std=0.02)
    dy = inputs.random_bf16((M, N), seed=seed + 2, std=1e-3)
    check_linear(x, w, dy, ("fprop", "dgrad", "wgrad"), seed)


@pytest.mark.parametrize("M", [1, 100, 300])
def test_token_counts_not_a_multiple_of_128(M):
    """Token tails: the last 128-row tile of fprop/dgrad is partial, the last
    128x1 token tile of the weight gradient's operands covers M % 128 tokens
    (padding tokens are zeros).  Every quantized byte and scale (padding
    included) and every GEMM output against the oracle."""
    N, K = 384, 256
    seed = 900 + M
    x = inputs.random_bf16((M, K), seed=seed)
    x[:, 7] *= 25.0
    w = inputs.random_bf16((N, K), seed=seed + 1, std=0.02)
    dy = inputs.random_bf16((M, N), seed=seed + 2, std=1e-3)
    check_linear(x, w, dy, ("fprop", "dgrad", "wgrad"), seed)


def test_persistent_tail_more_tiles_than_sms():
    # 148 SMs: 40 x 9 = 360 tiles of 128x256 -> every CTA loops, last wave partial.
    M, N, K = 5120, 2304, 256
    x = inputs.random_bf16((M, K), seed=5)
    w = inputs.random_bf16((N, K), seed=6, std=0.02)
    dy = inputs.random_bf16((M, N), seed=7, std=1e-3)
    check_linear(x, w, dy, ("fprop", "dgrad", "wgrad"), 5, sample=256)


def test_tiny_fprop_workload_full_output():
    wl = inputs.WORKLOADS["tiny_fprop_256x512x512"]
    d = inputs.make_linear_inputs(wl)[0]
    check_linear(d["x"], d["w"], None, ("fprop",), wl.seed)


@pytest.mark.parametrize("name", ["attn_qkv_fprop_8192x3072x2048", "mlp_gate_up_16384x11264x2048",
                                  "mlp_down_16384x2048x5632"])
def test_full_size_workloads_sampled_rows(name):
    wl = inputs.WORKLOADS[name]
    d = inputs.make_linear_inputs(wl)[0]
    check_linear(d["x"], d["w"], d.get("dy"), wl.linears[0].ops, wl.seed, sample=256)


def test_decoder_layer_workload_sampled_rows():
    wl = inputs.WORKLOADS["decoder_layer_32768"]
    for lin, d in zip(wl.linears, inputs.make_linear_inputs(wl)):
        check_linear(d["x"], d["w"], d["dy"], lin.ops, wl.seed, sample=256)
        torch.cuda.empty_cache()


def test_zero_inputs_give_zero_outputs():
    M, N, K = 256, 512, 256
    st = Fp8LinearStep(M, N, K)
    z = torch.zeros
    y, dx, dw = st.step(z(M, K, dtype=torch.bfloat16, device="cuda"), z(N, K, dtype=torch.bfloat16, device="cuda"),
                        z(M, N, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert not y.any() and not dx.any() and not dw.any()
    assert torch.all(st.sx == 1.0) and torch.all(st.sw == 1.0)


def test_deterministic():
    M, N, K = 1024, 1536, 768
    x = inputs.random_bf16((M, K), seed=11).cuda()
    w = inputs.random_bf16((N, K), seed=12, std=0.02).cuda()
    dy = inputs.random_bf16((M, N), seed=13, std=1e-3).cuda()
    st = Fp8LinearStep(M, N, K)
    a = [t.clone() for t in st.step(x, w, dy)]
    b = [t.clone() for t in st.step(x, w, dy)]
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int16), v.view(torch.int16))


def test_wgrad_split_k_is_deterministic_and_within_tolerance():
    """A weight gradient with few output tiles (2048 x 5632 -> 352 tiles of
    128 x 256 on 148 SMs) is split along the tokens; the split partials are
    added in a fixed order, so repeated runs are bitwise identical, and the
    result meets the acceptance rule like the unsplit one."""
    M, N, K = 8192, 2048, 5632
    assert B.fp8bs_gemm_wgrad_workspace_bytes(M, N, K) > 0, "this shape should split"
    x = inputs.random_bf16((M, K), seed=41)
    dy = inputs.random_bf16((M, N), seed=42, std=1e-3)
    _, _, xTq, sxT = B.fp8bs_quantize_act(x.cuda(), B.COLWISE_T)
    _, _, dyTq, sdyT = B.fp8bs_quantize_act(dy.cuda(), B.COLWISE_T)
    runs = [B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT).view(torch.int16).clone() for _ in range(5)]
    assert B.fp8bs_get_device_status() == 0
    for r in runs[1:]:
        assert torch.equal(r, runs[0])
    B.fp8bs_set_workspace(None)  # no scratch registered: the same call does not split
    unsplit = B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT, split=False)
    assert B.fp8bs_get_device_status() == 0
    rows = inputs.sample_rows(N, 4242, 256).numpy()
    oxTq, osxT = oracle.quant_colwise_128x1_T(x)
    odyTq, osdyT = oracle.quant_colwise_128x1_T(dy)
    acc, _, sab = oracle_gemm_rows("wgrad", odyTq, osdyT, oxTq, osxT, rows)
    split_bits = runs[0].cpu().numpy().view(np.uint16)[rows]
    assert_gemm_close(split_bits, acc, sab, "split wgrad")
    assert_gemm_close(np_bf16_bits(unsplit)[rows], acc, sab, "unsplit wgrad")


@pytest.mark.parametrize("op", ["fprop", "dgrad"])
def test_forward_and_data_gradient_tail_split(op):
    """2432 x 2048 outputs (152 tiles of 128 x 256 = one full wave on 148 SMs
    + 4 tiles), contraction 4096: the 4 tiles past the full wave (rows
    2304-2431, columns 1024-2047) are split in 4 parts.  Repeated runs are
    bitwise identical; the last 128 output rows and 64 random others meet the
    acceptance rule, with and without the split."""
    M, N, K = (2432, 2048, 4096) if op == "fprop" else (2432, 4096, 2048)
    code = B.OP_FPROP if op == "fprop" else B.OP_DGRAD
    assert B.fp8bs_gemm_workspace_bytes(code, M, N, K) > 0, "this shape should split"
    x = inputs.random_bf16((M, K), seed=81)
    w = inputs.random_bf16((N, K), seed=82, std=0.02)
    dy = inputs.random_bf16((M, N), seed=83, std=1e-3)
    wq, wqT, sw = B.fp8bs_quantize_weight(w.cuda(), want_t=True)
    if op == "fprop":
        aq, sa, _, _ = B.fp8bs_quantize_act(x.cuda(), B.ROWWISE)
        run = lambda split: B.fp8bs_gemm_fprop(aq, sa, wq, sw, split=split)
    else:
        aq, sa, _, _ = B.fp8bs_quantize_act(dy.cuda(), B.ROWWISE)
        run = lambda split: B.fp8bs_gemm_dgrad(aq, sa, wqT, sw, split=split)
    runs = [run(True).view(torch.int16).clone() for _ in range(3)]
    assert B.fp8bs_get_device_status() == 0
    for r in runs[1:]:
        assert torch.equal(r, runs[0])
    B.fp8bs_set_workspace(None)
    unsplit = run(False)
    assert B.fp8bs_get_device_status() == 0
    rows = np.concatenate([np.arange(M - 128, M), inputs.sample_rows(M - 128, 8181, 64).numpy()])
    owq, _, osw = oracle.quant_weight_128x128(w, want_t=False)
    if op == "fprop":
        oaq, osa = oracle.quant_rowwise_1x128(x)
        acc, _, sab = oracle_gemm_rows("fprop", oaq, osa, owq, osw, rows)
    else:
        oaq, osa = oracle.quant_rowwise_1x128(dy)
        acc, _, sab = oracle_gemm_rows("dgrad", oaq, osa, owq, osw, rows)
    assert_gemm_close(runs[0].cpu().numpy().view(np.uint16)[rows], acc, sab, f"split {op}")
    assert_gemm_close(np_bf16_bits(unsplit)[rows], acc, sab, f"unsplit {op}")


def test_tile_order_does_not_change_outputs():
    """The persistent CTAs' tile order (column strips of any width, the last
    one ragged, row-major, column by column) moves only which CTA computes
    a tile: unsplit products are bitwise equal in every order.  A product
    whose split plan splits every tile (uniform parts) is too, since no
    order changes which tiles are split."""
    M, N, K = 1000, 1792, 768   # 8 x 7 forward tiles, 8 x 3 data-gradient, 14 x 3 weight-gradient
    x = inputs.random_bf16((M, K), seed=311)
    x[:, 7] *= 25.0
    w = inputs.random_bf16((N, K), seed=312, std=0.02)
    dy = inputs.random_bf16((M, N), seed=313, std=1e-3)
    xq, sx, xTq, sxT = B.fp8bs_quantize_act(x.cuda(), B.ROWWISE | B.COLWISE_T)
    wq, wqT, sw = B.fp8bs_quantize_weight(w.cuda(), want_t=True)
    dyq, sdy, dyTq, sdyT = B.fp8bs_quantize_act(dy.cuda(), B.ROWWISE | B.COLWISE_T)
    Ms, Ns, Ks = 8192, 256, 512  # weight gradient of 2 x 2 tiles over 64 K blocks
    xs = inputs.random_bf16((Ms, Ks), seed=314)
    dys = inputs.random_bf16((Ms, Ns), seed=315, std=1e-3)
    _, _, xsTq, sxsT = B.fp8bs_quantize_act(xs.cuda(), B.COLWISE_T)
    _, _, dysTq, sdysT = B.fp8bs_quantize_act(dys.cuda(), B.COLWISE_T)
    plan = B.fp8bs_debug_split_plan(4, Ms // 128, torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["splits"] > 1 and plan["tail_first"] == 0, plan

    def run():
        outs = [B.fp8bs_gemm_fprop(xq, sx, wq, sw, split=False), B.fp8bs_gemm_dgrad(dyq, sdy, wqT, sw, split=False),
                B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT, split=False), B.fp8bs_gemm_wgrad(dysTq, sdysT, xsTq, sxsT)]
        assert B.fp8bs_get_device_status() == 0
        return [o.view(torch.int16).clone() for o in outs]

    ref = run()
    try:
        for strip in (1, 2, 3, 5, 64):
            B.fp8bs_debug_force_tile_order(strip)
            got = run()
            for name, a, b in zip(("fprop", "dgrad", "wgrad", "split wgrad"), got, ref):
                assert torch.equal(a, b), f"{name} differs with strips of {strip}"
    finally:
        B.fp8bs_debug_force_tile_order(0)
    oxq, osx = oracle.quant_rowwise_1x128(x)
    owq, _, osw = oracle.quant_weight_128x128(w, want_t=False)
    acc, _, sab = oracle_gemm_rows("fprop", oxq, osx, owq, osw, np.arange(M))
    assert_gemm_close(np_bf16_bits(ref[0].view(torch.bfloat16)), acc, sab, "fprop")


def test_grouped_launch_equals_single_launches():
    """Products of different shapes (a token tail, ragged output tiles) in
    one launch: forward and data-gradient products together, weight
    gradients in a group of their own.  Every output is bitwise equal to the
    member's own unsplit call; one member of each group is also checked
    against the oracle on all of its outputs."""
    B.fp8bs_set_workspace(None)  # single calls unsplit, like group members
    shapes = [(300, 384, 640), (1024, 1536, 768), (512, 256, 1280)]  # (tokens M, out N, in K)
    ops = []
    for i, (M, N, K) in enumerate(shapes):
        x = inputs.random_bf16((M, K), seed=90 + i)
        w = inputs.random_bf16((N, K), seed=95 + i, std=0.02)
        dy = inputs.random_bf16((M, N), seed=99 + i, std=1e-3)
        xq, sx, xTq, sxT = B.fp8bs_quantize_act(x.cuda(), B.ROWWISE | B.COLWISE_T)
        wq, wqT, sw = B.fp8bs_quantize_weight(w.cuda(), want_t=True)
        dyq, sdy, dyTq, sdyT = B.fp8bs_quantize_act(dy.cuda(), B.ROWWISE | B.COLWISE_T)
        ops.append(dict(x=x, w=w, dy=dy, xq=xq, sx=sx, xTq=xTq, sxT=sxT, wq=wq, wqT=wqT, sw=sw, dyq=dyq,
                        sdy=sdy, dyTq=dyTq, sdyT=sdyT))
    fwd = [(B.OP_FPROP, o["xq"], o["sx"], o["wq"], o["sw"], None) for o in ops] + \
          [(B.OP_DGRAD, ops[1]["dyq"], ops[1]["sdy"], ops[1]["wqT"], ops[1]["sw"], None)]
    wgt = [(B.OP_WGRAD, o["dyTq"], o["sdyT"], o["xTq"], o["sxT"], None) for o in ops]
    got_fwd = B.fp8bs_gemm_group(fwd)
    got_wgt = B.fp8bs_gemm_group(wgt)
    assert B.fp8bs_get_device_status() == 0
    single_fwd = [B.fp8bs_gemm_fprop(o["xq"], o["sx"], o["wq"], o["sw"], split=False) for o in ops] + \
                 [B.fp8bs_gemm_dgrad(ops[1]["dyq"], ops[1]["sdy"], ops[1]["wqT"], ops[1]["sw"], split=False)]
    single_wgt = [B.fp8bs_gemm_wgrad(o["dyTq"], o["sdyT"], o["xTq"], o["sxT"], split=False) for o in ops]
    assert B.fp8bs_get_device_status() == 0
    for g, s1 in zip(got_fwd + got_wgt, single_fwd + single_wgt):
        assert torch.equal(g.view(torch.int16), s1.view(torch.int16))
    o = ops[0]
    oxq, osx = oracle.quant_rowwise_1x128(o["x"])
    owq, _, osw = oracle.quant_weight_128x128(o["w"], want_t=False)
    acc, _, sab = oracle_gemm_rows("fprop", oxq, osx, owq, osw, np.arange(300))
    assert_gemm_close(np_bf16_bits(got_fwd[0]), acc, sab, "grouped fprop")
    oxTq, osxT = oracle.quant_colwise_128x1_T(o["x"])
    odyTq, osdyT = oracle.quant_colwise_128x1_T(o["dy"])
    acc, _, sab = oracle_gemm_rows("wgrad", odyTq, osdyT, oxTq, osxT, np.arange(384))
    assert_gemm_close(np_bf16_bits(got_wgt[0]), acc, sab, "grouped wgrad")


@pytest.mark.parametrize("M,N,K", [
    (300, 384, 640),      # token tail, ragged last column tile
    (2432, 2048, 4096),   # the last wave's tiles split in 4 (owners quantize after the fix-up)
    (8192, 3072, 2048),   # attention QKV forward at 8192 tokens
])
def test_fprop_with_fp8_output(M, N, K):
    """fp8bs_gemm_fprop_quant quantizes Y in the GEMM's epilogue.  Its BF16 Y
    equals fp8bs_gemm_fprop's bitwise; its E4M3 payload and scales equal the
    row-wise quantizer's on that BF16 Y bit for bit (the quantizer is pinned
    bit-exactly to the oracle by the quantizer tests), also when no BF16 Y is
    written; and the dequantized payload stays within the oracle product's
    tolerance plus one E4M3 rounding (|e| <= 2^-4 |v| above 2^-6 of the tile
    scale, <= 2^-10 of it below) on every output row of the first shape and
    on the last 128 rows (the split tiles of the second) + 64 seeded others
    of the larger two."""
    x = inputs.random_bf16((M, K), seed=7 + M)
    w = inputs.random_bf16((N, K), seed=8 + N, std=0.02)
    xq, sx, _, _ = B.fp8bs_quantize_act(x.cuda(), B.ROWWISE)
    wq, _, sw = B.fp8bs_quantize_weight(w.cuda(), want_t=False)
    y_plain = B.fp8bs_gemm_fprop(xq, sx, wq, sw)
    y, yq, sy = B.fp8bs_gemm_fprop_quant(xq, sx, wq, sw)
    _, yq2, sy2 = B.fp8bs_gemm_fprop_quant(xq, sx, wq, sw, want_bf16=False)
    assert B.fp8bs_get_device_status() == 0
    assert torch.equal(y.view(torch.int16), y_plain.view(torch.int16))
    q_ref, s_ref, _, _ = B.fp8bs_quantize_act(y, B.ROWWISE)
    assert torch.equal(yq, q_ref)
    assert torch.equal(sy.view(torch.int32), s_ref.view(torch.int32))
    assert torch.equal(yq2, yq) and torch.equal(sy2.view(torch.int32), sy.view(torch.int32))

    rows = np.arange(M) if M * N * K < 2 ** 34 else \
        np.concatenate([inputs.sample_rows(M - 128, 4343, 64).numpy(), np.arange(M - 128, M)])
    oxq, osx = oracle.quant_rowwise_1x128(x)
    owq, _, osw = oracle.quant_weight_128x128(w, want_t=False)
    acc, _, sab = oracle_gemm_rows("fprop", oxq, osx, owq, osw, rows)
    s_rows = np_f32(sy)[:, rows].T                                  # [rows][N/128]
    scale = np.repeat(s_rows, 128, axis=1).astype(np.float64)       # per element
    deq = oracle.e4m3_decode(np_u8(yq)[rows]) * scale
    ref = acc.astype(np.float64)
    gemm_tol = 2.0 ** -8 * np.abs(ref) + 1e-6 * sab
    bound = gemm_tol + 2.0 ** -4 * (np.abs(ref) + gemm_tol) + 2.0 ** -10 * scale
    assert np.all(np.abs(deq - ref) <= bound), float(np.max(np.abs(deq - ref) - bound))


@pytest.mark.parametrize("M,N,K", [(384, 256, 640), (8192, 2048, 5632)])
def test_wgrad_accumulates_in_fp32(M, N, K):
    """dW (FP32) += dY^T X, twice, starting from random FP32 values: every
    element equals D0 + k * acc up to the GEMM tolerance (no BF16 rounding
    here, so the 2^-8 |ref| term is generous) plus the FP32 adds' rounding;
    repeated from the same start it is bitwise reproducible.  The larger
    shape takes the split-K path."""
    x = inputs.random_bf16((M, K), seed=71)
    dy = inputs.random_bf16((M, N), seed=72, std=1e-3)
    _, _, xTq, sxT = B.fp8bs_quantize_act(x.cuda(), B.COLWISE_T)
    _, _, dyTq, sdyT = B.fp8bs_quantize_act(dy.cuda(), B.COLWISE_T)
    g = torch.Generator(device="cuda").manual_seed(73)
    d0 = torch.randn(N, K, generator=g, device="cuda") * 1e-3
    dw = d0.clone()
    B.fp8bs_gemm_wgrad_accumulate_f32(dyTq, sdyT, xTq, sxT, dw)
    once = dw.clone()
    B.fp8bs_gemm_wgrad_accumulate_f32(dyTq, sdyT, xTq, sxT, dw)
    assert B.fp8bs_get_device_status() == 0
    again = d0.clone()
    B.fp8bs_gemm_wgrad_accumulate_f32(dyTq, sdyT, xTq, sxT, again)
    assert torch.equal(again.view(torch.int32), once.view(torch.int32))
    rows = np.arange(N) if N * K <= 1 << 20 else inputs.sample_rows(N, 7474, 256).numpy()
    oxTq, osxT = oracle.quant_colwise_128x1_T(x)
    odyTq, osdyT = oracle.quant_colwise_128x1_T(dy)
    acc, _, sab = oracle_gemm_rows("wgrad", odyTq, osdyT, oxTq, osxT, rows)
    base = d0.cpu().numpy().astype(np.float64)[rows]
    acc = acc.astype(np.float64)
    for k, got in ((1, once), (2, dw)):
        ref = base + k * acc
        g64 = got.cpu().numpy().astype(np.float64)[rows]
        tol = k * (2.0 ** -8 * np.abs(acc) + 1e-6 * sab) + 2.0 ** -22 * (np.abs(ref) + np.abs(base))
        bad = np.abs(g64 - ref) > tol
        assert not bad.any(), f"accumulate x{k}: {int(bad.sum())} elements outside tolerance"


def test_bounded_wait_reports_timeout_and_gpu_stays_usable():
    """A withheld operand copy makes one CTA's MMA wait run out: the kernel
    records FP8BS_ERR_TIMEOUT and returns (no trap, no hang); the next
    launch on the same context is correct."""
    M, N, K = 512, 1024, 512
    x = inputs.random_bf16((M, K), seed=21)
    w = inputs.random_bf16((N, K), seed=22, std=0.02)
    xq, sx, _, _ = B.fp8bs_quantize_act(x.cuda(), B.ROWWISE)
    wq, _, sw = B.fp8bs_quantize_weight(w.cuda(), want_t=False)
    assert B.fp8bs_get_device_status() == 0
    try:
        B.fp8bs_debug_set_wait_timeout_ns(50_000_000)
        B.fp8bs_debug_set_fault(1)
        B.fp8bs_gemm_fprop(xq, sx, wq, sw)
        assert B.fp8bs_get_device_status() == 6  # FP8BS_ERR_TIMEOUT
    finally:
        B.fp8bs_debug_set_fault(0)
        B.fp8bs_debug_set_wait_timeout_ns(0)
    assert B.fp8bs_get_device_status() == 0
    y = B.fp8bs_gemm_fprop(xq, sx, wq, sw)
    assert B.fp8bs_get_device_status() == 0
    oxq, osx = oracle.quant_rowwise_1x128(x)
    owq, _, osw = oracle.quant_weight_128x128(w, want_t=False)
    acc, _, sab = oracle_gemm_rows("fprop", oxq, osx, owq, osw, np.arange(M))
    assert_gemm_close(np_bf16_bits(y), acc, sab, "fprop after timeout")


def test_rejects_bad_arguments():
    lib = B.load()
    t = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    p = t.data_ptr()
    assert lib.fp8bs_gemm_fprop(None, p, p, p, p, 128, 128, 128, None) == 1
    assert lib.fp8bs_gemm_fprop(p, p, p, p, p, 128, 100, 128, None) == 2
    assert lib.fp8bs_gemm_fprop(p, p, p, p, p, 0, 128, 128, None) == 2
    assert lib.fp8bs_gemm_wgrad(p, p, p, p, p, 128, 0, 128, None) == 2
    assert lib.fp8bs_gemm_dgrad(p + 8, p, p, p, p, 128, 128, 128, None) == 3


def test_long_contraction_full_output():
    """512 K blocks of promotion (K = 65536) on a small output, every
    element against the oracle; and the weight gradient over 65536 tokens."""
    M, N, K = 256, 512, 65536
    x = inputs.random_bf16((M, K), seed=51)
    w = inputs.random_bf16((N, K), seed=52, std=0.02)
    check_linear(x, w, None, ("fprop",), 51)
    Mt, Nt, Kt = 65536, 256, 256
    xt = inputs.random_bf16((Mt, Kt), seed=53)
    dyt = inputs.random_bf16((Mt, Nt), seed=54, std=1e-3)
    _, _, xTq, sxT = B.fp8bs_quantize_act(xt.cuda(), B.COLWISE_T)
    _, _, dyTq, sdyT = B.fp8bs_quantize_act(dyt.cuda(), B.COLWISE_T)
    dw = B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT)
    assert B.fp8bs_get_device_status() == 0
    # The 65536-token transposed operands bit for bit, then the oracle's GEMM
    # on its own quantization.
    oxTq, osxT = oracle.quant_colwise_128x1_T(xt)
    odyTq, osdyT = oracle.quant_colwise_128x1_T(dyt)
    same_bits(xTq, oxTq, "XTq over 65536 tokens")
    same_bits(sxT, osxT, "sXT over 65536 tokens")
    same_bits(dyTq, odyTq, "dYTq over 65536 tokens")
    same_bits(sdyT, osdyT, "sdYT over 65536 tokens")
    acc, _, sab = oracle_gemm_rows("wgrad", odyTq, osdyT, oxTq, osxT, np.arange(Nt))
    assert_gemm_close(np_bf16_bits(dw), acc, sab, "wgrad over 65536 tokens")


def test_tensor_map_cache_reuses_encoded_maps():
    """A repeated GEMM call on the same buffers takes every TMA tensor map
    from the cache (no driver encode) and gives the same bits; new buffers
    are encoded."""
    M, N, K = 512, 512, 512
    x = inputs.random_bf16((M, K), seed=71)
    w = inputs.random_bf16((N, K), seed=72, std=0.02)
    xq, sx, _, _ = B.fp8bs_quantize_act(x.cuda(), B.ROWWISE)
    wq, _, sw = B.fp8bs_quantize_weight(w.cuda(), want_t=False)
    y1 = B.fp8bs_gemm_fprop(xq, sx, wq, sw)
    e1 = B.load().fp8bs_debug_tensor_map_encodes()
    y2 = torch.empty_like(y1)
    B.fp8bs_gemm_fprop(xq, sx, wq, sw, y=y2)
    e2 = B.load().fp8bs_debug_tensor_map_encodes()
    B.fp8bs_gemm_fprop(xq, sx, wq, sw, y=y2)
    assert B.load().fp8bs_debug_tensor_map_encodes() == e2   # all maps cached
    assert e2 - e1 == 1                                        # only y2's store map was new
    assert B.fp8bs_get_device_status() == 0
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_split_wgrad_completes_while_other_work_holds_most_sms():
    """The parts of a split tile never wait for each other: with 100 SMs held
    for 0.5 s by another stream's kernel, so that most of the GEMM's CTAs
    start only afterwards, and the device wait limit cut to 0.1 s, a split
    weight gradient still completes with FP8BS_OK and the same bits as an
    undisturbed run (a part that waited for a part not yet resident would
    hit the limit)."""
    M, N, K = 8192, 2048, 5632
    assert B.fp8bs_gemm_wgrad_workspace_bytes(M, N, K) > 0, "this shape should split"
    x = inputs.random_bf16((M, K), seed=141)
    dy = inputs.random_bf16((M, N), seed=142, std=1e-3)
    _, _, xTq, sxT = B.fp8bs_quantize_act(x.cuda(), B.COLWISE_T)
    _, _, dyTq, sdyT = B.fp8bs_quantize_act(dy.cuda(), B.COLWISE_T)
    ref = B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT)
    assert B.fp8bs_get_device_status() == 0
    lib = B.load()
    busy, work = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    try:
        assert lib.fp8bs_debug_set_wait_timeout_ns(100_000_000) == 0
        assert lib.fp8bs_debug_occupy_sms(100, 500_000_000, busy.cuda_stream) == 0
        with torch.cuda.stream(work):
            out = B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT, stream=work)
        assert B.fp8bs_get_device_status(work) == 0
        torch.cuda.synchronize()
    finally:
        lib.fp8bs_debug_set_wait_timeout_ns(0)
    assert B.fp8bs_get_device_status() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_grouped_weight_gradients_split_like_single_calls():
    """Weight gradients that split on their own split the same way inside a
    group (each in its own region of the scratch): every output equals the
    member's own split call bit for bit, and meets the rule on sampled rows."""
    shapes = [(8192, 2048, 5632), (8192, 256, 512), (2048, 384, 256)]   # (tokens, N, K): tail split, uniform, whole
    members, singles, data = [], [], []
    for i, (M, N, K) in enumerate(shapes):
        x = inputs.random_bf16((M, K), seed=150 + i)
        dy = inputs.random_bf16((M, N), seed=160 + i, std=1e-3)
        _, _, xTq, sxT = B.fp8bs_quantize_act(x.cuda(), B.COLWISE_T)
        _, _, dyTq, sdyT = B.fp8bs_quantize_act(dy.cuda(), B.COLWISE_T)
        members.append((B.OP_WGRAD, dyTq, sdyT, xTq, sxT, None))
        data.append((x, dy))
    assert B.fp8bs_gemm_wgrad_workspace_bytes(*shapes[0]) > 0 and B.fp8bs_gemm_wgrad_workspace_bytes(*shapes[1]) > 0
    got = B.fp8bs_gemm_group(members)
    for (_, dyTq, sdyT, xTq, sxT, _) in members:
        singles.append(B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT))
    assert B.fp8bs_get_device_status() == 0
    for g, s1 in zip(got, singles):
        assert torch.equal(g.view(torch.int16), s1.view(torch.int16))
    x, dy = data[1]
    oxTq, osxT = oracle.quant_colwise_128x1_T(x)
    odyTq, osdyT = oracle.quant_colwise_128x1_T(dy)
    acc, _, sab = oracle_gemm_rows("wgrad", odyTq, osdyT, oxTq, osxT, np.arange(256))
    assert_gemm_close(np_bf16_bits(got[1]), acc, sab, "grouped split wgrad")
