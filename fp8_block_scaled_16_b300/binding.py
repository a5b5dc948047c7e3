"""Python binding of the C ABI in include/fp8bs.h (ctypes, argument
marshalling only).

Each function has the name of the C entry point it calls.  It takes torch
CUDA tensors, allocates any output the caller did not pass (torch is the
device-memory allocator here), passes raw device pointers and the current
CUDA stream to the library, and raises Fp8bsError on a non-OK status.  All
arithmetic runs in the library's kernels; there is no fallback path: if the
library is missing or the device is not an sm_103 GPU, the call fails.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import build as _build

ROWWISE = 1
COLWISE_T = 2
OP_FPROP, OP_DGRAD, OP_WGRAD = 0, 1, 2   # fp8bs_gemm_workspace_bytes products
DEBUG_F32_OUT = 1                        # fp8bs_debug_set_flags: FP32 accumulator outputs
_debug_flags = 0

STATUS = {
    0: "FP8BS_OK", 1: "FP8BS_ERR_INVALID_ARG", 2: "FP8BS_ERR_SHAPE", 3: "FP8BS_ERR_ALIGN",
    4: "FP8BS_ERR_ARCH", 5: "FP8BS_ERR_LAUNCH", 6: "FP8BS_ERR_TIMEOUT", 7: "FP8BS_ERR_CUDA",
}

# Every symbol include/fp8bs.h declares, with its ctypes signature.
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
class GemmArgs(ctypes.Structure):
    """fp8bs_gemm_args: one member of a grouped GEMM."""
    _fields_ = [("op", ctypes.c_int), ("a", ctypes.c_void_p), ("sa", ctypes.c_void_p), ("b", ctypes.c_void_p),
                ("sb", ctypes.c_void_p), ("out", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64)]


GROUP_MAX = 4  # FP8BS_GROUP_MAX

SIGNATURES = {
    "fp8bs_quantize_act": (ctypes.c_int, [_P, _I64, _I64, ctypes.c_uint, _P, _P, _P, _P, _P]),
    "fp8bs_quantize_weight": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P, _P]),
    "fp8bs_gemm_fprop": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "fp8bs_gemm_dgrad": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "fp8bs_gemm_fprop_quant": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "fp8bs_gemm_fprop_swiglu_quant": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "fp8bs_debug_silu_mul": (ctypes.c_int, [_P, _P, _I64, _P, _P]),
    "fp8bs_gemm_wgrad": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "fp8bs_get_device_status": (ctypes.c_int, [_P]),
    "fp8bs_set_workspace": (ctypes.c_int, [_P, _I64]),
    "fp8bs_gemm_workspace_bytes": (_I64, [ctypes.c_int, _I64, _I64, _I64]),
    "fp8bs_gemm_group": (ctypes.c_int, [ctypes.POINTER(GemmArgs), ctypes.c_int, _P]),
    "fp8bs_debug_split_plan": (ctypes.c_int, [_I64, _I64, ctypes.c_int, _P]),
    "fp8bs_debug_tile_order": (ctypes.c_int, [_I64, _I64, _I64, ctypes.c_int32, _I64, _I64, _I64, ctypes.c_int32,
                                              _P]),
    "fp8bs_gemm_wgrad_workspace_bytes": (_I64, [_I64, _I64, _I64]),
    "fp8bs_gemm_wgrad_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "fp8bs_gemm_wgrad_accumulate_f32": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "fp8bs_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fp8bs_launch_count": (_I64, []),
    "fp8bs_debug_tensor_map_encodes": (_I64, []),
    "fp8bs_debug_set_wait_timeout_ns": (ctypes.c_int, [_I64]),
    "fp8bs_debug_set_fault": (ctypes.c_int, [ctypes.c_int]),
    "fp8bs_debug_force_tile_order": (ctypes.c_int, [ctypes.c_int]),
    "fp8bs_debug_set_flags": (ctypes.c_int, [ctypes.c_uint]),
    "fp8bs_debug_occupy_sms": (ctypes.c_int, [ctypes.c_int, _I64, _P]),
    "fp8bs_debug_e4m3_encode_bits": (ctypes.c_int, [ctypes.c_uint32, _I64, _P, _P]),
}


class Fp8bsError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = status


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libfp8bs.so (built in-tree by build.py).  Raises if it is
    missing: there is no other implementation to fall back to."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with `python -m fp8_block_scaled_16_b300.build`")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise Fp8bsError(rc, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, dtype, shape, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _out(t: Optional[torch.Tensor], shape, dtype, device) -> torch.Tensor:
    return torch.empty(shape, dtype=dtype, device=device) if t is None else t


def _gemm_out_dtype():
    """BF16, or FP32 while the FP32-output test mode is on."""
    return torch.float32 if _debug_flags & DEBUG_F32_OUT else torch.bfloat16


# ---------------------------------------------------------------- entry points

def padded_tokens(rows: int) -> int:
    """Leading dimension of token-major arrays: rows rounded up to 128."""
    return (rows + 127) // 128 * 128


def fp8bs_quantize_act(x: torch.Tensor, flags: int = ROWWISE, q=None, s=None, qT=None, sT=None,
                       stream=None) -> Tuple[Optional[torch.Tensor], ...]:
    """x BF16 [rows][cols] -> (q u8 [rows][cols], s f32 [cols/128][Mp],
    qT u8 [cols][Mp], sT f32 [Mp/128][cols]) with Mp = rows rounded up to 128;
    the pair for a layout that `flags` does not request is (None, None)."""
    rows, cols = x.shape
    mp = padded_tokens(rows)
    dev = x.device
    xp = _dev(x, torch.bfloat16, (rows, cols), "x")
    ptrs = [None, None, None, None]
    if flags & ROWWISE:
        q = _out(q, (rows, cols), torch.uint8, dev)
        s = _out(s, (cols // 128, mp), torch.float32, dev)
        ptrs[0] = _dev(q, torch.uint8, (rows, cols), "q")
        ptrs[1] = _dev(s, torch.float32, (cols // 128, mp), "s")
    else:
        q = s = None
    if flags & COLWISE_T:
        qT = _out(qT, (cols, mp), torch.uint8, dev)
        sT = _out(sT, (mp // 128, cols), torch.float32, dev)
        ptrs[2] = _dev(qT, torch.uint8, (cols, mp), "qT")
        ptrs[3] = _dev(sT, torch.float32, (mp // 128, cols), "sT")
    else:
        qT = sT = None
    _check(load().fp8bs_quantize_act(xp, rows, cols, flags, *ptrs, _stream(stream)), "fp8bs_quantize_act")
    return q, s, qT, sT


def fp8bs_quantize_weight(w: torch.Tensor, q=None, qT=None, s=None, want_t: bool = True, stream=None):
    """w BF16 [n][k] -> (q u8 [n][k], qT u8 [k][n] or None, s f32 [n/128][k/128])."""
    n, k = w.shape
    dev = w.device
    wp = _dev(w, torch.bfloat16, (n, k), "w")
    q = _out(q, (n, k), torch.uint8, dev)
    s = _out(s, (n // 128, k // 128), torch.float32, dev)
    if want_t:
        qT = _out(qT, (k, n), torch.uint8, dev)
    qTp = _dev(qT, torch.uint8, (k, n), "qT") if qT is not None else None
    _check(load().fp8bs_quantize_weight(wp, n, k, _dev(q, torch.uint8, (n, k), "q"), qTp,
                                        _dev(s, torch.float32, (n // 128, k // 128), "s"), _stream(stream)),
           "fp8bs_quantize_weight")
    return q, qT, s


def fp8bs_gemm_fprop(xq, sx, wq, sw, y=None, stream=None, split=True) -> torch.Tensor:
    """Y [M][N] BF16 = X W^T from Xq [M][K], sx [K/128][Mp], Wq [N][K], sw [N/128][K/128].
    With split=True the binding makes sure split-K scratch is registered."""
    M, K = xq.shape
    N = wq.shape[0]
    if split:
        _ensure_workspace(OP_FPROP, M, N, K, xq.device)
    y = _out(y, (M, N), _gemm_out_dtype(), xq.device)
    _check(load().fp8bs_gemm_fprop(
        _dev(xq, torch.uint8, (M, K), "xq"), _dev(sx, torch.float32, (K // 128, padded_tokens(M)), "sx"),
        _dev(wq, torch.uint8, (N, K), "wq"), _dev(sw, torch.float32, (N // 128, K // 128), "sw"),
        _dev(y, _gemm_out_dtype(), (M, N), "y"), M, N, K, _stream(stream)), "fp8bs_gemm_fprop")
    return y


def fp8bs_gemm_fprop_quant(xq, sx, wq, sw, y=None, yq=None, sy=None, want_bf16=True, stream=None, split=True):
    """Y = X W^T with Y's 1x128 row-wise quantization done in the GEMM's
    epilogue.  Returns (y or None, yq u8 [M][N], sy f32 [N/128][Mp]); yq/sy
    equal fp8bs_quantize_act(y, ROWWISE)."""
    M, K = xq.shape
    N = wq.shape[0]
    if split:
        _ensure_workspace(OP_FPROP, M, N, K, xq.device)
    y = _out(y, (M, N), torch.bfloat16, xq.device) if want_bf16 else None
    yq = _out(yq, (M, N), torch.uint8, xq.device)
    sy = _out(sy, (N // 128, padded_tokens(M)), torch.float32, xq.device)
    _check(load().fp8bs_gemm_fprop_quant(
        _dev(xq, torch.uint8, (M, K), "xq"), _dev(sx, torch.float32, (K // 128, padded_tokens(M)), "sx"),
        _dev(wq, torch.uint8, (N, K), "wq"), _dev(sw, torch.float32, (N // 128, K // 128), "sw"),
        _dev(y, torch.bfloat16, (M, N), "y") if y is not None else None,
        _dev(yq, torch.uint8, (M, N), "yq"), _dev(sy, torch.float32, (N // 128, padded_tokens(M)), "sy"),
        M, N, K, _stream(stream)), "fp8bs_gemm_fprop_quant")
    return y, yq, sy


def fp8bs_gemm_fprop_swiglu_quant(xq, sx, wq, sw, h=None, hq=None, sh=None, want_bf16=True, stream=None,
                                  split=True):
    """H = SiLU(X Wg^T) * (X Wu^T) from the gate+up weight interleaved in
    128-row blocks (see interleave_gate_up in linear.py), with H's 1x128
    quantization.  Returns (h or None, hq u8 [M][I], sh f32 [I/128][Mp])."""
    M, K = xq.shape
    N2 = wq.shape[0]
    I = N2 // 2
    if split:
        _ensure_workspace(OP_FPROP, M, N2, K, xq.device)
    h = _out(h, (M, I), torch.bfloat16, xq.device) if want_bf16 else None
    hq = _out(hq, (M, I), torch.uint8, xq.device)
    sh = _out(sh, (I // 128, padded_tokens(M)), torch.float32, xq.device)
    _check(load().fp8bs_gemm_fprop_swiglu_quant(
        _dev(xq, torch.uint8, (M, K), "xq"), _dev(sx, torch.float32, (K // 128, padded_tokens(M)), "sx"),
        _dev(wq, torch.uint8, (N2, K), "wq"), _dev(sw, torch.float32, (N2 // 128, K // 128), "sw"),
        _dev(h, torch.bfloat16, (M, I), "h") if h is not None else None,
        _dev(hq, torch.uint8, (M, I), "hq"), _dev(sh, torch.float32, (I // 128, padded_tokens(M)), "sh"),
        M, N2, K, _stream(stream)), "fp8bs_gemm_fprop_swiglu_quant")
    return h, hq, sh


def fp8bs_debug_silu_mul(g: torch.Tensor, u: torch.Tensor, h=None, stream=None) -> torch.Tensor:
    """h = bf16(SiLU(g) * u) elementwise for BF16 CUDA tensors of one shape."""
    h = _out(h, tuple(g.shape), torch.bfloat16, g.device)
    _dev(u, torch.bfloat16, tuple(g.shape), "u")
    _check(load().fp8bs_debug_silu_mul(_dev(g, torch.bfloat16, tuple(g.shape), "g"), u.data_ptr(), g.numel(),
                                       _dev(h, torch.bfloat16, tuple(g.shape), "h"), _stream(stream)),
           "fp8bs_debug_silu_mul")
    return h


def fp8bs_gemm_dgrad(dyq, sdy, wqT, sw, dx=None, stream=None, split=True) -> torch.Tensor:
    """dX [M][K] BF16 = dY W from dYq [M][N], sdy [N/128][Mp], WqT [K][N], sw [N/128][K/128].
    With split=True the binding makes sure split-K scratch is registered."""
    M, N = dyq.shape
    K = wqT.shape[0]
    if split:
        _ensure_workspace(OP_DGRAD, M, N, K, dyq.device)
    dx = _out(dx, (M, K), _gemm_out_dtype(), dyq.device)
    _check(load().fp8bs_gemm_dgrad(
        _dev(dyq, torch.uint8, (M, N), "dyq"), _dev(sdy, torch.float32, (N // 128, padded_tokens(M)), "sdy"),
        _dev(wqT, torch.uint8, (K, N), "wqT"), _dev(sw, torch.float32, (N // 128, K // 128), "sw"),
        _dev(dx, _gemm_out_dtype(), (M, K), "dx"), M, N, K, _stream(stream)), "fp8bs_gemm_dgrad")
    return dx


_workspaces = {}  # device index -> registered scratch tensor


def _ensure_workspace(op: int, M: int, N: int, K: int, device) -> None:
    """Registers (torch-allocated) scratch for the split-K path of product
    `op` if this shape would use more than the device has registered."""
    _ensure_workspace_bytes(int(load().fp8bs_gemm_workspace_bytes(op, M, N, K)), device)


def _ensure_workspace_bytes(need: int, device) -> None:
    """Registers at least `need` bytes of scratch on `device`.  A new buffer
    replaces the old one only after the device is idle."""
    if need <= 0:
        return
    idx = device.index if device.index is not None else torch.cuda.current_device()
    cur = _workspaces.get(idx)
    if cur is not None and cur.numel() >= need:
        return
    with torch.cuda.device(idx):
        torch.cuda.synchronize()
        buf = torch.empty(need, dtype=torch.uint8, device=torch.device("cuda", idx))
        _check(load().fp8bs_set_workspace(buf.data_ptr(), need), "fp8bs_set_workspace")
    _workspaces[idx] = buf


def fp8bs_set_workspace(ws: Optional[torch.Tensor]) -> None:
    """Registers a uint8 CUDA tensor as the current device's scratch (None
    unregisters)."""
    if ws is None:
        _check(load().fp8bs_set_workspace(None, 0), "fp8bs_set_workspace")
        _workspaces.pop(torch.cuda.current_device(), None)
        return
    _check(load().fp8bs_set_workspace(_dev(ws, torch.uint8, (ws.numel(),), "ws"), ws.numel()),
           "fp8bs_set_workspace")
    _workspaces[ws.device.index] = ws


def fp8bs_gemm_workspace_bytes(op: int, M: int, N: int, K: int) -> int:
    return int(load().fp8bs_gemm_workspace_bytes(op, M, N, K))


def fp8bs_gemm_wgrad_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().fp8bs_gemm_wgrad_workspace_bytes(M, N, K))


def fp8bs_gemm_wgrad(dyTq, sdyT, xTq, sxT, dw=None, stream=None, split=True) -> torch.Tensor:
    """dW [N][K] BF16 = dY^T X from dYTq [N][Mp], sdyT [Mp/128][N], XTq [K][Mp], sxT [Mp/128][K]
    (Mp: the token count rounded up to 128; the padding tokens are zero payloads).
    With split=True the binding makes sure split-K scratch is registered."""
    N, M = dyTq.shape
    K = xTq.shape[0]
    if split:
        _ensure_workspace(OP_WGRAD, M, N, K, dyTq.device)
    dw = _out(dw, (N, K), _gemm_out_dtype(), dyTq.device)
    _check(load().fp8bs_gemm_wgrad(
        _dev(dyTq, torch.uint8, (N, M), "dyTq"), _dev(sdyT, torch.float32, (M // 128, N), "sdyT"),
        _dev(xTq, torch.uint8, (K, M), "xTq"), _dev(sxT, torch.float32, (M // 128, K), "sxT"),
        _dev(dw, _gemm_out_dtype(), (N, K), "dw"), M, N, K, _stream(stream)), "fp8bs_gemm_wgrad")
    return dw


def fp8bs_gemm_wgrad_accumulate_f32(dyTq, sdyT, xTq, sxT, dw, stream=None) -> torch.Tensor:
    """dW (FP32 [N][K], updated in place) += dY^T X."""
    N, M = dyTq.shape
    K = xTq.shape[0]
    _ensure_workspace(OP_WGRAD, M, N, K, dyTq.device)
    _check(load().fp8bs_gemm_wgrad_accumulate_f32(
        _dev(dyTq, torch.uint8, (N, M), "dyTq"), _dev(sdyT, torch.float32, (M // 128, N), "sdyT"),
        _dev(xTq, torch.uint8, (K, M), "xTq"), _dev(sxT, torch.float32, (M // 128, K), "sxT"),
        _dev(dw, torch.float32, (N, K), "dw"), M, N, K, _stream(stream)), "fp8bs_gemm_wgrad_accumulate_f32")
    return dw


def fp8bs_gemm_wgrad_noalloc(dyTq, sdyT, xTq, sxT, dw=None, stream=None) -> torch.Tensor:
    """As fp8bs_gemm_wgrad, but the library takes its split-K scratch from a
    static device array instead of registered memory (for callers that
    cannot allocate); shapes that need more scratch raise Fp8bsError."""
    N, M = dyTq.shape
    K = xTq.shape[0]
    dw = _out(dw, (N, K), torch.bfloat16, dyTq.device)
    _check(load().fp8bs_gemm_wgrad_noalloc(
        _dev(dyTq, torch.uint8, (N, M), "dyTq"), _dev(sdyT, torch.float32, (M // 128, N), "sdyT"),
        _dev(xTq, torch.uint8, (K, M), "xTq"), _dev(sxT, torch.float32, (M // 128, K), "sxT"),
        _dev(dw, torch.bfloat16, (N, K), "dw"), M, N, K, _stream(stream)), "fp8bs_gemm_wgrad_noalloc")
    return dw


def fp8bs_get_device_status(stream=None) -> int:
    return int(load().fp8bs_get_device_status(_stream(stream)))


def fp8bs_status_string(status: int) -> str:
    return load().fp8bs_status_string(status).decode()


def fp8bs_launch_count() -> int:
    return int(load().fp8bs_launch_count())


def fp8bs_debug_set_wait_timeout_ns(ns: int) -> None:
    _check(load().fp8bs_debug_set_wait_timeout_ns(ns), "fp8bs_debug_set_wait_timeout_ns")


def fp8bs_debug_set_flags(flags: int) -> None:
    """Test modes of the GEMMs (DEBUG_F32_OUT: fprop / dgrad / wgrad write
    their FP32 accumulators; the wrappers then allocate float32 outputs);
    0 turns them off."""
    global _debug_flags
    _check(load().fp8bs_debug_set_flags(flags), "fp8bs_debug_set_flags")
    _debug_flags = flags


def fp8bs_debug_force_tile_order(strip: int) -> None:
    """Test hook: GEMMs take tiles in column strips `strip` wide (0: the
    library's own choice per shape)."""
    _check(load().fp8bs_debug_force_tile_order(strip), "fp8bs_debug_force_tile_order")


def fp8bs_debug_set_fault(mode: int) -> None:
    _check(load().fp8bs_debug_set_fault(mode), "fp8bs_debug_set_fault")


def fp8bs_debug_e4m3_encode_bits(first: int, n: int, out: Optional[torch.Tensor] = None, stream=None):
    out = _out(out, (n,), torch.uint8, torch.device("cuda"))
    _check(load().fp8bs_debug_e4m3_encode_bits(first, n, _dev(out, torch.uint8, (n,), "out"), _stream(stream)),
           "fp8bs_debug_e4m3_encode_bits")
    return out


def fp8bs_debug_split_plan(tiles: int, kblocks: int, sms: int) -> dict:
    """The library's split-K plan for a product of `tiles` output tiles and
    `kblocks` contraction blocks on `sms` SMs (host computation only)."""
    out = (ctypes.c_int64 * 4)()
    _check(load().fp8bs_debug_split_plan(tiles, kblocks, sms, ctypes.cast(out, ctypes.c_void_p)),
           "fp8bs_debug_split_plan")
    return {"splits": out[0], "tail_first": out[1], "units": out[2], "bytes": out[3]}


def fp8bs_debug_tile_order(m_tiles: int, n_tiles: int, kc: int, splits: int = 1, tail_first: int = 0,
                           grid: int = 148, l2_bytes: int = 126 << 20, out_bytes: int = 2) -> dict:
    """The tile order a GEMM launch would take (host computation only):
    column-strip width (== n_tiles: row-major) and the estimated DRAM bytes
    of operand panels for that order and for row-major."""
    out = (ctypes.c_int64 * 3)()
    _check(load().fp8bs_debug_tile_order(m_tiles, n_tiles, kc, splits, tail_first, grid, l2_bytes, out_bytes,
                                         ctypes.cast(out, ctypes.c_void_p)), "fp8bs_debug_tile_order")
    return {"strip": out[0], "dram_bytes": out[1], "row_major_dram_bytes": out[2]}


def fp8bs_gemm_group(members, stream=None, split=True):
    """Several products in one launch.  `members` lists (op, a, sa, b, sb,
    out) with op OP_FPROP (a = Xq, sa = sx, b = Wq, sb = sw), OP_DGRAD (dYq,
    sdy, WqT, sw) or OP_WGRAD (dYTq, sdyT, XTq, sxT), operand layouts as for
    that op's own function; `out` may be None (allocated).  Forward and
    data-gradient products may share a group, weight gradients group alone.
    Returns the outputs in order.  With split=True the binding registers
    scratch for every member's split plan, so each output equals the op's
    own call (split=True) bit for bit; without scratch each equals the op's
    unsplit result."""
    if not 1 <= len(members) <= GROUP_MAX:
        raise ValueError(f"a group has 1..{GROUP_MAX} members, got {len(members)}")
    arr = (GemmArgs * len(members))()
    outs = []
    need = 0
    for i, (op, a, sa, b, sb, out) in enumerate(members):
        if op == OP_FPROP:
            (M, K), N = a.shape, b.shape[0]
            shapes = ((M, K), (K // 128, padded_tokens(M)), (N, K), (N // 128, K // 128), (M, N))
        elif op == OP_DGRAD:
            (M, N), K = a.shape, b.shape[0]
            shapes = ((M, N), (N // 128, padded_tokens(M)), (K, N), (N // 128, K // 128), (M, K))
        elif op == OP_WGRAD:
            (N, Mp), K = a.shape, b.shape[0]
            M = Mp
            shapes = ((N, Mp), (Mp // 128, N), (K, Mp), (Mp // 128, K), (N, K))
        else:
            raise ValueError(f"unknown op {op}")
        out = _out(out, shapes[4], torch.bfloat16, a.device)
        arr[i] = GemmArgs(op, _dev(a, torch.uint8, shapes[0], "a"), _dev(sa, torch.float32, shapes[1], "sa"),
                          _dev(b, torch.uint8, shapes[2], "b"), _dev(sb, torch.float32, shapes[3], "sb"),
                          _dev(out, torch.bfloat16, shapes[4], "out"), M, N, K)
        need += max(0, int(load().fp8bs_gemm_workspace_bytes(op, M, N, K)))
        outs.append(out)
    if split and need > 0:
        _ensure_workspace_bytes(need, members[0][1].device)
    _check(load().fp8bs_gemm_group(arr, len(members), _stream(stream)), "fp8bs_gemm_group")
    return outs
