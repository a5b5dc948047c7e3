"""The weight gradient for callers that cannot allocate device memory.

fp8bs_gemm_wgrad_noalloc computes the same dW = dY^T X as fp8bs_gemm_wgrad
but takes its split-K scratch from a static device array inside the library
instead of a caller-registered buffer, for callers (plug-ins into a framework
that owns all device memory, latency-critical loops that cannot afford a
cudaMalloc) that have no allocator to offer.  These tests call it through the
C ABI and compare it with the regular entry point.  The file is named so that
pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_16_b300 import binding as B
from fp8_block_scaled_16_b300 import inputs
from tests._parity import assert_gemm_close, np_bf16_bits, oracle_gemm_rows

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 48 << 20  # FP8BS_NOALLOC_SCRATCH_BYTES in include/fp8bs.h


def _quantized_pair(M, N, K, seed):
    x = inputs.random_bf16((M, K), seed=seed)
    dy = inputs.random_bf16((M, N), seed=seed + 1, std=1e-3)
    _, _, xTq, sxT = B.fp8bs_quantize_act(x.cuda(), B.COLWISE_T)
    _, _, dyTq, sdyT = B.fp8bs_quantize_act(dy.cuda(), B.COLWISE_T)
    return x, dy, xTq, sxT, dyTq, sdyT


def test_noalloc_wgrad_matches_the_regular_entry_point_on_two_calls():
    """Both entry points take the same split plan and add the parts' partial
    sums in the same fixed order, so the no-allocation result must equal the
    regular one bit for bit, on every output and on each of two calls in a
    row (the second call finds the first call's contents in the shared
    array); sampled rows are also checked against the oracle."""
    assert torch.cuda.is_available()
    lib = B.load()
    # 2048 x 5632 outputs = 352 tiles of 128 x 256 (2 full waves on 148 SMs
    # + 56 tiles): the last 56 tiles' tokens are split in two across CTAs,
    # which needs ~7 MiB of scratch.
    M, N, K = 8192, 2048, 5632
    need = B.fp8bs_gemm_wgrad_workspace_bytes(M, N, K)
    assert 0 < need <= SCRATCH_BYTES
    x, dy, xTq, sxT, dyTq, sdyT = _quantized_pair(M, N, K, seed=61)
    regular = B.fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT)
    assert B.fp8bs_get_device_status() == 0
    rows = inputs.sample_rows(N, 6161, 256).numpy()
    oxTq, osxT = oracle.quant_colwise_128x1_T(x)
    odyTq, osdyT = oracle.quant_colwise_128x1_T(dy)
    acc, _, sumabs = oracle_gemm_rows("wgrad", odyTq, osdyT, oxTq, osxT, rows)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full((N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lib.fp8bs_gemm_wgrad_noalloc(dyTq.data_ptr(), sdyT.data_ptr(), xTq.data_ptr(), sxT.data_ptr(),
                                          out.data_ptr(), M, N, K, stream)
        assert rc == 0, B.fp8bs_status_string(rc)
        assert B.fp8bs_get_device_status() == 0
        assert torch.equal(out.view(torch.int16), regular.view(torch.int16)), f"call {call + 1}: bits differ"
        assert_gemm_close(np_bf16_bits(out)[rows], acc, sumabs, f"no-alloc wgrad, call {call + 1}")


def test_noalloc_wgrad_rejects_shapes_that_need_more_scratch():
    lib = B.load()
    # 3968 x 2048 outputs = 248 tiles (1.7 waves on 148 SMs): every tile split
    # four ways, ~93 MiB of scratch.
    M, N, K = 16384, 3968, 2048
    assert B.fp8bs_gemm_wgrad_workspace_bytes(M, N, K) > SCRATCH_BYTES
    dyTq = torch.zeros(N, M, dtype=torch.uint8, device="cuda")
    xTq = torch.zeros(K, M, dtype=torch.uint8, device="cuda")
    sdyT = torch.ones(M // 128, N, device="cuda")
    sxT = torch.ones(M // 128, K, device="cuda")
    out = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    launches = B.fp8bs_launch_count()
    rc = lib.fp8bs_gemm_wgrad_noalloc(dyTq.data_ptr(), sdyT.data_ptr(), xTq.data_ptr(), sxT.data_ptr(),
                                      out.data_ptr(), M, N, K, torch.cuda.current_stream().cuda_stream)
    assert rc == 2  # FP8BS_ERR_SHAPE
    assert B.fp8bs_launch_count() == launches
    assert not out.any()
