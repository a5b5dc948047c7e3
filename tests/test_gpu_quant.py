"""GPU parity of the quantizers against the oracle: payload bytes and scales
must be bit-identical, through the C ABI."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_16_b300 import binding as B
from fp8_block_scaled_16_b300 import inputs
from tests._parity import THREADS, np_f32, np_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    B.load()
    yield
    torch.cuda.synchronize()


def check_rowwise(x: torch.Tensor):
    q, s, _, _ = B.fp8bs_quantize_act(x.cuda(), B.ROWWISE)
    oq, os_ = oracle.quant_rowwise_1x128(x)
    assert np.array_equal(np_u8(q), oq), "1x128 payload differs"
    assert np.array_equal(np_f32(s).view(np.uint32), os_.view(np.uint32)), "1x128 scales differ"


def check_colwise(x: torch.Tensor, fused: bool):
    flags = B.COLWISE_T | (B.ROWWISE if fused else 0)
    q, s, qT, sT = B.fp8bs_quantize_act(x.cuda(), flags)
    oqT, osT = oracle.quant_colwise_128x1_T(x)
    assert np.array_equal(np_u8(qT), oqT), "128x1 transposed payload differs"
    assert np.array_equal(np_f32(sT).view(np.uint32), osT.view(np.uint32)), "128x1 scales differ"
    if fused:
        oq, os_ = oracle.quant_rowwise_1x128(x)
        assert np.array_equal(np_u8(q), oq)
        assert np.array_equal(np_f32(s).view(np.uint32), os_.view(np.uint32))


def check_weight(w: torch.Tensor):
    q, qT, s = B.fp8bs_quantize_weight(w.cuda())
    oq, oqT, os_ = oracle.quant_weight_128x128(w)
    assert np.array_equal(np_u8(q), oq), "weight payload differs"
    assert np.array_equal(np_u8(qT), oqT), "transposed weight payload differs"
    assert np.array_equal(np_f32(s).view(np.uint32), os_.view(np.uint32)), "weight scales differ"
    q2, none, s2 = B.fp8bs_quantize_weight(w.cuda(), want_t=False)
    assert none is None and torch.equal(q2, q) and torch.equal(s2, s)


def test_encoder_matches_oracle_on_all_fp32_patterns():
    """The kernels' FP32->E4M3 conversion against the oracle's hand-written
    encoder on all 2^32 bit patterns (NaNs compared as 'any NaN code')."""
    chunk = 1 << 28
    out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    for c in range(16):
        first = c * chunk
        B.fp8bs_debug_e4m3_encode_bits(first, chunk, out)
        gpu = np_u8(out)
        parts = np.array_split(np.arange(chunk, dtype=np.int64), THREADS)
        with ThreadPoolExecutor(THREADS) as ex:
            ref = np.concatenate(list(ex.map(lambda p: oracle.e4m3_encode_bits(first + int(p[0]), p.size), parts)))
        bits = np.arange(chunk, dtype=np.uint32) + np.uint32(first)
        nan_in = (bits & 0x7FFFFFFF) > 0x7F800000
        same = gpu == ref
        same |= nan_in & ((gpu & 0x7F) == 0x7F) & ((ref & 0x7F) == 0x7F)
        if not same.all():
            i = int(np.argmin(same))
            raise AssertionError(f"pattern {int(bits[i]):#010x}: gpu {int(gpu[i]):#04x} oracle {int(ref[i]):#04x}")


def test_rowwise_small_shapes_and_edge_tiles():
    x = inputs.random_bf16((384, 640), seed=101)
    x[0, :128] = 0.0                       # all-zero tile
    x[1, 128:256] = -0.0                   # all negative-zero tile
    x[2, :128] = 0.0
    x[2, 7] = -(2.0 ** -133)               # amax: smallest BF16 subnormal
    x[3, 256:384] *= 1e30                  # huge values
    x[4, 384:512] *= 1e-38                 # subnormal-scale values
    x[5, 5] = 3.0e38                       # near BF16 max
    x[6, :] = 448.0                        # constant tile
    x[:, 300] *= 60.0                      # outlier channel
    check_rowwise(x)


def test_colwise_and_fused_small_shapes_and_edge_tiles():
    x = inputs.random_bf16((384, 640), seed=102)
    x[:128, 0] = 0.0
    x[128:256, 1] = -0.0
    x[:128, 2] = 0.0
    x[77, 2] = 2.0 ** -133
    x[:, 3] *= 1e30
    x[:, 600] *= 1e-38
    x[300, :] *= 50.0
    check_colwise(x, fused=False)
    check_colwise(x, fused=True)


@pytest.mark.parametrize("rows", [1, 100, 129, 300])
def test_token_tails_bit_exact(rows):
    """Token counts that are not a multiple of 128, both layouts fused and
    alone: payloads and scales (with the padding) equal the oracle's."""
    x = inputs.random_bf16((rows, 384), seed=500 + rows)
    x[:, 11] *= 45.0
    check_rowwise(x)
    check_colwise(x, fused=False)
    check_colwise(x, fused=True)


def test_weight_small_shapes_and_edge_blocks():
    w = inputs.random_bf16((384, 640), seed=103, std=0.02)
    w[:128, :128] = 0.0
    w[128:256, 128:256] *= 1e-36
    w[300, 600] = 5.0
    check_weight(w)


def test_tiny_fprop_workload_quantizers():
    d = inputs.make_linear_inputs(inputs.WORKLOADS["tiny_fprop_256x512x512"])[0]
    check_rowwise(d["x"])
    check_colwise(d["x"], fused=True)
    check_weight(d["w"])


@pytest.mark.parametrize("name", ["attn_qkv_fprop_8192x3072x2048", "mlp_gate_up_16384x11264x2048",
                                  "mlp_down_16384x2048x5632"])
def test_full_size_workload_quantizers(name):
    wl = inputs.WORKLOADS[name]
    d = inputs.make_linear_inputs(wl)[0]
    lin = wl.linears[0]
    if "wgrad" in lin.ops:
        check_colwise(d["x"], fused=True)
    else:
        check_rowwise(d["x"])
    check_weight(d["w"])
    if "dy" in d:
        if "wgrad" in lin.ops:
            check_colwise(d["dy"], fused=True)
        else:
            check_rowwise(d["dy"])


def test_deterministic_and_rejects_bad_arguments():
    x = inputs.random_bf16((256, 256), seed=104).cuda()
    a = B.fp8bs_quantize_act(x, B.ROWWISE | B.COLWISE_T)
    b = B.fp8bs_quantize_act(x, B.ROWWISE | B.COLWISE_T)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    with pytest.raises(B.Fp8bsError) as e:
        B.fp8bs_quantize_act(inputs.random_bf16((256, 200), seed=1).cuda(), B.ROWWISE)
    assert e.value.status == 2
    lib = B.load()
    assert lib.fp8bs_quantize_act(x.data_ptr() + 2, 256, 256, 1, a[0].data_ptr(), a[1].data_ptr(),
                                  None, None, None) == 3
    assert lib.fp8bs_quantize_act(x.data_ptr(), 256, 256, 0, None, None, None, None, None) == 1


def test_largest_grid_checked_by_row_block_slices():
    """The largest activation the launch geometry allows (65535 row blocks of
    128 tokens, one 128-column block: 2.1 GB of BF16).  Quantization is local
    to each 128x128 tile, so any row block of the output must equal the
    oracle run on that row block alone: the first, the last and some seeded
    ones in between are checked, in both layouts."""
    rows, cols = 65535 * 128, 128
    g = torch.Generator(device="cuda").manual_seed(77)
    x = torch.randn(rows, cols, generator=g, device="cuda").to(torch.bfloat16)
    x[:, 5] *= 40.0
    q, s, qT, sT = B.fp8bs_quantize_act(x, B.ROWWISE | B.COLWISE_T)
    # The row-wise layout alone (its own kernel) gives the same bytes.
    q1, s1, _, _ = B.fp8bs_quantize_act(x, B.ROWWISE)
    torch.cuda.synchronize()
    assert torch.equal(q1, q) and torch.equal(s1.view(torch.int32), s.view(torch.int32))
    del q1, s1
    blocks = [0, 1, 65534] + inputs.sample_rows(65535, 99, 13).tolist()
    for b in sorted(set(blocks)):
        xs = x[b * 128:(b + 1) * 128].cpu()
        oq, os_ = oracle.quant_rowwise_1x128(xs)
        oqT, osT = oracle.quant_colwise_128x1_T(xs)
        assert np.array_equal(np_u8(q[b * 128:(b + 1) * 128]), oq), b
        assert np.array_equal(np_f32(s[:, b * 128:(b + 1) * 128]).view(np.uint32), os_.view(np.uint32)), b
        assert np.array_equal(np_u8(qT[:, b * 128:(b + 1) * 128]), oqT), b
        assert np.array_equal(np_f32(sT[b:b + 1]).view(np.uint32), osT.view(np.uint32)), b
    del x, q, s, qT, sT
    torch.cuda.empty_cache()
