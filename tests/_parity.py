"""Shared helpers for the parity tests: run the oracle on row samples in
parallel threads (the C oracle releases the GIL), move tensors between the
GPU and numpy, and apply the GEMM acceptance rule."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle

THREADS = max(1, min(64, os.cpu_count() or 1))


def np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def np_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def oracle_gemm_rows(kind: str, a, sa, b, sb, rows):
    """Oracle GEMM on the listed output rows, split across threads."""
    fn = {"fprop": oracle.gemm_fprop, "dgrad": oracle.gemm_dgrad, "wgrad": oracle.gemm_wgrad}[kind]
    rows = np.asarray(rows, dtype=np.int64)
    chunks = [c for c in np.array_split(rows, min(THREADS, max(1, rows.size))) if c.size]
    with ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        parts = list(ex.map(lambda r: fn(a, sa, b, sb, rows=r), chunks))
    return tuple(np.concatenate([p[i] for p in parts], axis=0) for i in range(3))


def assert_gemm_close(gpu_bf16_bits: np.ndarray, ref_acc: np.ndarray, sumabs: np.ndarray, what: str):
    """Acceptance rule for GEMM outputs:
        |gpu - ref| <= 2^-8 |ref| + 1e-6 sum_k |a_k b_k|
    with ref the oracle's FP32 accumulator before BF16 rounding and the sum
    over the dequantized operands.  The 2^-8 |ref| term covers the BF16
    rounding of the output (at most half a BF16 ulp, <= 2^-8 of the value);
    the second term covers the tensor core's own summation order inside each
    128-wide block."""
    g = bf16_bits_to_f64(gpu_bf16_bits)
    r = ref_acc.astype(np.float64)
    tol = 2.0 ** -8 * np.abs(r) + 1e-6 * sumabs
    err = np.abs(g - r)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(i)}: gpu={g[tuple(i)]!r} ref={r[tuple(i)]!r} tol={tol[tuple(i)]:.3g}"
                           for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outputs outside tolerance; {detail}")
    return float((err / np.maximum(tol, 1e-300)).max())
