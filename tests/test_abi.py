"""The C ABI library loads without a GPU and exports every symbol that
include/fp8bs.h declares; argument validation answers before any launch.
(No call here reaches a kernel: every call fails validation first.)"""
import ctypes
import os
import re
import subprocess

import pytest

from fp8_block_scaled_16_b300 import binding as B
from fp8_block_scaled_16_b300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(fp8bs_\w+)\s*\(", text))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fp8bs_quantize_act", "fp8bs_quantize_weight", "fp8bs_gemm_fprop", "fp8bs_gemm_dgrad",
              "fp8bs_gemm_wgrad", "fp8bs_get_device_status", "fp8bs_status_string"):
        assert n in names
    assert names == set(B.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.check_output(["nm", "-D", "--defined-only", build_mod.LIB], text=True)
    exported = set(re.findall(r"\bT (fp8bs_\w+)", out))
    assert declared_functions() <= exported
    for n in declared_functions():
        assert hasattr(lib, n)


def test_library_needs_no_driver_to_load():
    out = subprocess.check_output(["ldd", build_mod.LIB], text=True)
    assert "libcuda.so" not in out  # the driver API is resolved at run time


def test_status_strings(lib):
    for code, name in B.STATUS.items():
        assert B.fp8bs_status_string(code) == name
    assert B.fp8bs_status_string(99) == "FP8BS_ERR_UNKNOWN"


def test_validation_before_launch(lib):
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: every call below fails validation
    odd = ctypes.c_void_p(0x10008)
    assert lib.fp8bs_quantize_act(None, 128, 128, 1, fake, fake, None, None, None) == 1
    assert lib.fp8bs_quantize_act(fake, 128, 128, 0, fake, fake, None, None, None) == 1
    assert lib.fp8bs_quantize_act(fake, 128, 128, 4, fake, fake, None, None, None) == 1
    assert lib.fp8bs_quantize_act(fake, 128, 128, 2, fake, fake, None, None, None) == 1  # qT/sT missing
    assert lib.fp8bs_quantize_act(fake, 128, 100, 1, fake, fake, None, None, None) == 2   # features % 128
    assert lib.fp8bs_quantize_act(fake, 0, 128, 1, fake, fake, None, None, None) == 2     # no tokens
    assert lib.fp8bs_quantize_act(fake, 128, -128, 1, fake, fake, None, None, None) == 2
    assert lib.fp8bs_quantize_act(fake, 128 * 65536, 128, 1, fake, fake, None, None, None) == 2
    assert lib.fp8bs_quantize_act(odd, 128, 128, 1, fake, fake, None, None, None) == 3
    assert lib.fp8bs_quantize_weight(fake, 128, 128, None, None, fake, None) == 1
    assert lib.fp8bs_quantize_weight(fake, 128, 130, fake, None, fake, None) == 2
    assert lib.fp8bs_quantize_weight(fake, 128, 128, fake, odd, fake, None) == 3
    for fn in (lib.fp8bs_gemm_fprop, lib.fp8bs_gemm_dgrad, lib.fp8bs_gemm_wgrad):
        assert fn(fake, fake, None, fake, fake, 128, 128, 128, None) == 1
        assert fn(fake, fake, fake, fake, fake, 128, 256, 0, None) == 2
        assert fn(fake, fake, fake, fake, fake, 0, 256, 128, None) == 2     # no tokens
        assert fn(fake, fake, fake, fake, fake, -5, 256, 128, None) == 2
        assert fn(fake, fake, fake, fake, fake, 128, 200, 128, None) == 2
        assert fn(fake, fake, fake, odd, fake, 128, 128, 128, None) == 3
    fq = lib.fp8bs_gemm_fprop_quant
    assert fq(fake, fake, fake, fake, None, fake, None, 128, 256, 128, None) == 1      # no scales for Yq
    assert fq(fake, fake, fake, fake, None, None, fake, 128, 256, 128, None) == 1      # no Yq
    assert fq(fake, fake, fake, fake, None, fake, fake, 128, 200, 128, None) == 2
    assert fq(fake, fake, fake, fake, None, odd, fake, 128, 256, 128, None) == 3
    assert fq(fake, fake, fake, fake, odd, fake, fake, 128, 256, 128, None) == 3       # optional Y misaligned
    assert fq(fake, fake, fake, fake, None, fake, odd, 128, 256, 128, None) == 3
    fs = lib.fp8bs_gemm_fprop_swiglu_quant
    assert fs(fake, fake, fake, fake, None, fake, None, 128, 256, 128, None) == 1      # no scales for Hq
    assert fs(fake, fake, fake, fake, None, fake, fake, 128, 384, 128, None) == 2      # N2 not a multiple of 256
    assert fs(fake, fake, fake, fake, odd, fake, fake, 128, 256, 128, None) == 3
    assert lib.fp8bs_debug_silu_mul(None, fake, 16, fake, None) == 1
    assert lib.fp8bs_debug_silu_mul(fake, fake, -1, fake, None) == 1
    assert lib.fp8bs_debug_e4m3_encode_bits(0, 16, None, None) == 1
    assert lib.fp8bs_debug_e4m3_encode_bits(0xFFFFFFF0, 32, fake, None) == 2
    assert lib.fp8bs_debug_e4m3_encode_bits(0, 16, odd, None) == 3
    assert lib.fp8bs_set_workspace(None, 5) == 1
    assert lib.fp8bs_set_workspace(fake, -1) == 1
    assert lib.fp8bs_set_workspace(fake, 1000) == 1               # below the 64 KiB flag region
    assert lib.fp8bs_set_workspace(ctypes.c_void_p(0x10010), 1 << 20) == 3
    assert lib.fp8bs_gemm_wgrad_workspace_bytes(0, 128, 128) == -2
    assert lib.fp8bs_gemm_wgrad_workspace_bytes(100, 100, 128) == -2
    assert lib.fp8bs_gemm_wgrad_workspace_bytes(128, 0, 128) == -2


def test_group_validation_before_launch(lib):
    fake = 0x10000
    good = B.GemmArgs(B.OP_FPROP, fake, fake, fake, fake, fake, 128, 256, 128)
    wgrad = B.GemmArgs(B.OP_WGRAD, fake, fake, fake, fake, fake, 128, 256, 128)
    bad_op = B.GemmArgs(7, fake, fake, fake, fake, fake, 128, 256, 128)
    bad_shape = B.GemmArgs(B.OP_DGRAD, fake, fake, fake, fake, fake, 128, 200, 128)
    null_out = B.GemmArgs(B.OP_FPROP, fake, fake, fake, fake, None, 128, 256, 128)
    odd = B.GemmArgs(B.OP_FPROP, fake, fake, fake + 8, fake, fake, 128, 256, 128)

    def call(*members, count=None):
        arr = (B.GemmArgs * max(1, len(members)))(*members)
        return lib.fp8bs_gemm_group(arr, len(members) if count is None else count, None)

    assert lib.fp8bs_gemm_group(None, 1, None) == 1
    assert call(good, count=0) == 1
    assert call(good, good, good, good, good) == 1              # more than FP8BS_GROUP_MAX
    assert call(good, bad_op) == 1
    assert call(good, wgrad) == 1                               # weight gradients group alone
    assert call(good, null_out) == 1
    assert call(bad_shape) == 2
    assert call(good, odd) == 3
    assert lib.fp8bs_gemm_workspace_bytes(9, 128, 256, 128) == -1   # unknown product
    assert lib.fp8bs_gemm_workspace_bytes(B.OP_FPROP, 0, 256, 128) == -2


def test_debug_setters(lib):
    assert lib.fp8bs_debug_set_fault(2) == 1
    assert lib.fp8bs_debug_set_fault(0) == 0
    assert lib.fp8bs_debug_set_wait_timeout_ns(-1) == 1
    assert lib.fp8bs_debug_set_wait_timeout_ns(0) == 0
    assert lib.fp8bs_launch_count() >= 0


C_CONSUMER = r"""
#include <stdio.h>
#include <string.h>
#include "fp8bs.h"

int main(void) {
    /* argument checks answer before any device work, so this runs without a GPU */
    int64_t plan[4];
    fp8bs_gemm_args g;
    memset(&g, 0, sizeof g);
    g.op = FP8BS_OP_FPROP;
    if (fp8bs_gemm_fprop(NULL, NULL, NULL, NULL, NULL, 128, 256, 128, NULL) != FP8BS_ERR_INVALID_ARG) return 1;
    if (fp8bs_quantize_act((const void*)0x10000, 128, 100, FP8BS_ROWWISE, (uint8_t*)0x10000, (float*)0x10000,
                           NULL, NULL, NULL) != FP8BS_ERR_SHAPE) return 2;
    if (fp8bs_gemm_group(&g, 0, NULL) != FP8BS_ERR_INVALID_ARG) return 3;
    if (fp8bs_debug_split_plan(768, 64, 148, plan) != FP8BS_OK || plan[0] != 5 || plan[1] != 740) return 4;
    if (strcmp(fp8bs_status_string(FP8BS_OK), "FP8BS_OK") != 0) return 5;
    printf("ok\n");
    return 0;
}
"""


def test_header_is_plain_c_and_the_library_links(tmp_path, lib):
    """A C program (gcc, C11, no C++) includes the header, links the library
    and gets the documented answers from calls that fail validation."""
    src = tmp_path / "consumer.c"
    src.write_text(C_CONSUMER)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(build_mod.LIB)
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                           "-L", libdir, "-lfp8bs", f"-Wl,-rpath,{libdir}", "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.strip() == "ok", (out.returncode, out.stdout, out.stderr)
