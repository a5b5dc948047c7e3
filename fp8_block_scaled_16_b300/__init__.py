"""FP8 fine-grained block-quantized linear layer for NVIDIA B300 (sm_103a).

The compute lives in the CUDA library ``libfp8bs.so`` (C ABI:
``include/fp8bs.h``); ``binding`` marshals torch tensors to it, ``linear``
chains the calls into one linear layer's forward and backward step (also as
a torch autograd op and module), and
``inputs`` draws the seeded synthetic workloads.  Importing the package does
not load the library; the first call does, and fails if it is missing.
"""
from __future__ import annotations

import importlib

_BINDING_NAMES = (
    "ROWWISE", "COLWISE_T", "Fp8bsError",
    "fp8bs_quantize_act", "fp8bs_quantize_weight", "fp8bs_gemm_fprop", "fp8bs_gemm_dgrad",
    "fp8bs_gemm_fprop_quant", "fp8bs_gemm_fprop_swiglu_quant", "fp8bs_debug_silu_mul",
    "fp8bs_gemm_wgrad", "fp8bs_get_device_status", "fp8bs_status_string", "fp8bs_launch_count",
    "fp8bs_debug_set_wait_timeout_ns", "fp8bs_debug_set_fault", "fp8bs_debug_e4m3_encode_bits",
    "fp8bs_debug_split_plan",
    "fp8bs_set_workspace", "fp8bs_gemm_workspace_bytes", "fp8bs_gemm_wgrad_workspace_bytes",
    "fp8bs_gemm_wgrad_noalloc", "OP_FPROP", "OP_DGRAD", "OP_WGRAD", "fp8bs_gemm_group", "GemmArgs",
    "fp8bs_gemm_wgrad_accumulate_f32",
)

_LINEAR_NAMES = ("Fp8LinearStep", "Fp8LinearFunction", "Fp8Linear")

__all__ = list(_BINDING_NAMES) + list(_LINEAR_NAMES)


def __getattr__(name):
    if name in _BINDING_NAMES:
        return getattr(importlib.import_module(".binding", __name__), name)
    if name in _LINEAR_NAMES:
        return getattr(importlib.import_module(".linear", __name__), name)
    raise AttributeError(name)
