// act.cuh -- SwiGLU activation of a gate+up projection's outputs.
//
// h = SiLU(g) * u with SiLU(g) = g / (1 + e^-g), evaluated in FP32 on the
// BF16 values of the gate and up outputs and rounded to BF16: the
// activation between a decoder layer's gate+up and down projections, whose
// result is the down projection's FP8 input.  The pages keep activations
// out of the FP8 path; this is its BF16-in, BF16-out form, one rounding per
// operation so that any IEEE implementation of the same steps gives the
// same bits.
//
// e^x: Cody-Waite reduction (W. J. Cody, W. Waite, "Software Manual for the
// Elementary Functions", 1980).  x = n ln2 + r, n = rint(x log2 e), r from a
// two-part ln 2 whose high part has 16 significant bits (n * high part is
// exact); e^r by its degree-7 Taylor polynomial in Horner form with fused
// multiply-adds; times 2^n.  Inputs above 88 give +Inf, below -87 give 0,
// so 2^n stays a normal power of two.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace fp8bs {

__device__ __forceinline__ float exp_cw(float x) {
    if (x > 88.0f) return __int_as_float(0x7f800000);
    if (x < -87.0f) return 0.0f;
    const float n = rintf(__fmul_rn(x, 1.44269502f));             // log2(e) in FP32
    float r = __fmaf_rn(-n, 0.693145751953125f, x);               // ln 2, high part: 45426 / 2^16
    r = __fmaf_rn(-n, 1.42860677e-06f, r);                        // ln 2 - high part
    float p = 1.0f / 5040.0f;
    p = __fmaf_rn(p, r, 1.0f / 720.0f);
    p = __fmaf_rn(p, r, 1.0f / 120.0f);
    p = __fmaf_rn(p, r, 1.0f / 24.0f);
    p = __fmaf_rn(p, r, 1.0f / 6.0f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __fmul_rn(p, __int_as_float((static_cast<int>(n) + 127) << 23));
}

// FP32 h = SiLU(g) * u for BF16-valued g and u (before the final rounding).
__device__ __forceinline__ float silu_mul_f32(float g, float u) {
    const float d = __fadd_rn(1.0f, exp_cw(-g));
    return __fmul_rn(__fdiv_rn(g, d), u);
}

// The same as a called function: the GEMM epilogue evaluates it for 128
// values per thread, and 128 inlined copies would crowd the instruction
// cache that the K-block loop runs from.
__device__ __noinline__ float silu_mul_call(float g, float u) { return silu_mul_f32(g, u); }

// Test kernel: h[i] = bf16(SiLU(g[i]) * u[i]) on BF16 bit patterns.
__global__ void silu_mul_kernel(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* h) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float v = silu_mul_f32(__uint_as_float(static_cast<uint32_t>(g[i]) << 16),
                                     __uint_as_float(static_cast<uint32_t>(u[i]) << 16));
        h[i] = static_cast<uint16_t>(f32x2_to_bf16x2(v, 0.0f) & 0xFFFFu);
    }
}

}  // namespace fp8bs
