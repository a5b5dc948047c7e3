"""CPU oracle for the FP8 fine-grained block-quantized linear layer.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline / reference leg may import this package.
The product library never loads it and shares no code with it.

The arithmetic lives in plain C (``fp8bs_oracle.c``), compiled single
threaded with ``-O2 -fno-fast-math -ffp-contract=off``.  This module only
compiles it, loads it with ctypes and marshals numpy arrays.

Pinned by ``tests/test_oracle_*.py`` (CPU only):
  * E4M3 decode: a hand-made table of codes whose values the OCP FP8
    definition fixes, and PyTorch's own float8_e4m3fn decoder on all 256
    codes;
  * E4M3 encode: PyTorch's float8_e4m3fn cast on every FP32 bit pattern in
    the non-saturating range, round trips of all codes, midpoint (tie) cases;
  * quantizers: hand-derived tiles, invariants (the amax element maps to
    +-448, power-of-two equivariance, W/W^T byte identity, the dequantization
    error bound, the all-zero tile);
  * GEMMs: integer brute force of one 128^3 block, a float64 GEMM of the
    dequantized operands within the analytic promotion bound, the unit-scale
    special case, and the fprop/dgrad/wgrad transposition identities;
  * SwiGLU activation (tests/test_oracle_activation.py): its exponential
    within 1 ulp of float64 e^x, SiLU(g)*u within one BF16 ulp of the
    float64 formula on every BF16 g in [-24, 24], and its special cases.
tests/test_oracle_mutants.py plants one plausible mistake at a time in a
copy of the C source and checks that some pin fails.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8bs_oracle.c")
_LIB = os.path.join(_HERE, "liborc_fp8bs.so")
_CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11"]
SOURCE, CFLAGS = _SRC, _CFLAGS  # for tests that compile altered copies

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc) next to its source; returns the .so path.
    Test hook: FP8BS_ORACLE_LIB names a library built elsewhere from a
    deliberately altered copy of the source (tests/test_oracle_mutants.py),
    which the pins must then reject."""
    alt = os.environ.get("FP8BS_ORACLE_LIB")
    if alt:
        return alt
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


_P = ctypes.c_void_p
_I = ctypes.c_int64
_SIGS = {
    "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
    "orc_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
    "orc_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
    "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
    "orc_quant_rowwise_1x128": (None, [_P, _I, _I, _P, _P]),
    "orc_quant_colwise_128x1_T": (None, [_P, _I, _I, _P, _P]),
    "orc_quant_weight_128x128": (None, [_P, _I, _I, _P, _P, _P]),
    "orc_gemm_fprop": (None, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _P, _P]),
    "orc_gemm_dgrad": (None, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _P, _P]),
    "orc_gemm_wgrad": (None, [_P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _P, _P]),
    "orc_e4m3_encode_array": (None, [_P, _I, _P]),
    "orc_e4m3_encode_bits": (None, [ctypes.c_uint32, _I, _P]),
    "orc_e4m3_decode_array": (None, [_P, _I, _P]),
    "orc_exp_cw": (ctypes.c_float, [ctypes.c_float]),
    "orc_silu_mul_bf16": (ctypes.c_uint16, [ctypes.c_uint16, ctypes.c_uint16]),
    "orc_silu_mul_array": (None, [_P, _P, _I, _P]),
    "orc_exp_cw_array": (None, [_P, _I, _P]),
}


def lib():
    global _lib
    with _lock:
        if _lib is None:
            l = ctypes.CDLL(build())
            for name, (res, args) in _SIGS.items():
                f = getattr(l, name)
                f.restype = res
                f.argtypes = args
            _lib = l
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(x) -> np.ndarray:
    """Accept a uint16 array of BF16 bit patterns or a torch bfloat16 tensor."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # only for marshalling a CPU bf16 tensor's bits

    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


# ---------------------------------------------------------------- formats

def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().orc_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_array(_ptr(f), f.size, _ptr(out))
    return out


def e4m3_encode_bits(first: int, n: int) -> np.ndarray:
    """Encode the FP32 values whose bit patterns are first .. first+n-1."""
    out = np.empty(n, dtype=np.uint8)
    lib().orc_e4m3_encode_bits(ctypes.c_uint32(first), n, _ptr(out))
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(v: float) -> int:
    return int(lib().orc_f32_to_bf16(ctypes.c_float(v)))


# ---------------------------------------------------------------- quantizers

def padded_tokens(rows: int) -> int:
    """Token count rounded up to whole 128-token blocks (the leading dimension
    of token-major arrays)."""
    return (rows + 127) // 128 * 128


def quant_rowwise_1x128(x):
    """x BF16 [rows][cols] -> (q u8 [rows][cols], s f32 [cols/128][Mp]);
    Mp = rows rounded up to 128, padding rows' scales are 1."""
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((cols // 128, padded_tokens(rows)), np.float32)
    lib().orc_quant_rowwise_1x128(_ptr(xb), rows, cols, _ptr(q), _ptr(s))
    return q, s


def quant_colwise_128x1_T(x):
    """x BF16 [rows][cols] -> (qT u8 [cols][Mp], sT f32 [Mp/128][cols]);
    padding tokens have payload 0."""
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    mp = padded_tokens(rows)
    qT = np.empty((cols, mp), np.uint8)
    sT = np.empty((mp // 128, cols), np.float32)
    lib().orc_quant_colwise_128x1_T(_ptr(xb), rows, cols, _ptr(qT), _ptr(sT))
    return qT, sT


def quant_weight_128x128(w, want_t: bool = True):
    """w BF16 [n][k] -> (q u8 [n][k], qT u8 [k][n] or None, s f32 [n/128][k/128])."""
    wb = _bf16_bits(w)
    n, k = wb.shape
    q = np.empty((n, k), np.uint8)
    qT = np.empty((k, n), np.uint8) if want_t else None
    s = np.empty((n // 128, k // 128), np.float32)
    lib().orc_quant_weight_128x128(_ptr(wb), n, k, _ptr(q),
                                   _ptr(qT) if want_t else None, _ptr(s))
    return q, qT, s


# ---------------------------------------------------------------- GEMMs

def _rows_arg(rows, total):
    if rows is None:
        rows = np.arange(total, dtype=np.int64)
    return np.ascontiguousarray(rows, dtype=np.int64)


def _gemm(fn, a, sa, b, sb, M, N, K, rows, out_len, total_rows, ld=None):
    r = _rows_arg(rows, total_rows)
    acc = np.empty((r.size, out_len), np.float32)
    bf = np.empty((r.size, out_len), np.uint16)
    sab = np.empty((r.size, out_len), np.float64)
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    extra = () if ld is None else (ld,)
    fn(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), M, N, K, *extra, _ptr(r), r.size,
       _ptr(acc), _ptr(bf), _ptr(sab))
    return acc, bf, sab


def gemm_fprop(xq, sx, wq, sw, rows=None):
    """Y = X W^T.  Returns (acc f32 unrounded, y bf16 bits, sum|ab| f64) for
    the listed rows of Y ([len(rows)][N])."""
    M, K = xq.shape
    N = wq.shape[0]
    assert sx.shape[0] == K // 128 and sx.shape[1] >= M
    return _gemm(lib().orc_gemm_fprop, xq, sx, wq, sw, M, N, K, rows, N, M, ld=sx.shape[1])


def gemm_dgrad(dyq, sdy, wq, sw, rows=None):
    """dX = dY W, with W given in its forward layout Wq [N][K]."""
    M, N = dyq.shape
    K = wq.shape[1]
    assert sdy.shape[0] == N // 128 and sdy.shape[1] >= M
    return _gemm(lib().orc_gemm_dgrad, dyq, sdy, wq, sw, M, N, K, rows, K, M, ld=sdy.shape[1])


def gemm_wgrad(dytq, sdyt, xtq, sxt, rows=None):
    """dW = dY^T X from the token-major transposed payloads ([features][Mp],
    zero padding tokens included).  rows index dW's rows (output features n)."""
    N, M = dytq.shape
    K = xtq.shape[0]
    return _gemm(lib().orc_gemm_wgrad, dytq, sdyt, xtq, sxt, M, N, K, rows, K, N)



# ---------------------------------------------------------------- activation

def exp_cw(x: np.ndarray) -> np.ndarray:
    """e^x in FP32 by Cody-Waite reduction and a degree-7 Taylor polynomial."""
    v = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(v.shape, np.float32)
    lib().orc_exp_cw_array(_ptr(v), v.size, _ptr(out))
    return out


def silu_mul(g, u) -> np.ndarray:
    """h = SiLU(g) * u elementwise on BF16 bit patterns (uint16 arrays or
    bf16 tensors of one shape); returns BF16 bits."""
    gb, ub = _bf16_bits(g), _bf16_bits(u)
    assert gb.shape == ub.shape
    out = np.empty(gb.shape, np.uint16)
    lib().orc_silu_mul_array(_ptr(gb), _ptr(ub), gb.size, _ptr(out))
    return out
