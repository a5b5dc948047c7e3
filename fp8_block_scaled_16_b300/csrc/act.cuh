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

// e^x of two values with packed FP32 operations; each lane of a packed
// multiply or fused multiply-add rounds like the scalar operation, so every
// lane follows the scalar steps: n = rint(x log2 e) (log2 e rounded to
// FP32), r = x - n ln2 in two fused steps (ln 2's high part 45426 / 2^16,
// then the rest), the degree-7 Taylor polynomial of e^r in Horner form, and
// the product with 2^n.  Lanes above 88 give +Inf, below -87 give 0; they
// are evaluated on the clamped value, whose result is then replaced.
__device__ __forceinline__ float2 exp_cw2(float2 x) {
    const float2 xc = make_float2(fminf(fmaxf(x.x, -87.0f), 88.0f), fminf(fmaxf(x.y, -87.0f), 88.0f));
    const float2 m = __fmul2_rn(xc, make_float2(1.44269502f, 1.44269502f));
    const float2 n = make_float2(rintf(m.x), rintf(m.y));
    const float2 nn = make_float2(-n.x, -n.y);
    float2 r = __ffma2_rn(nn, make_float2(0.693145751953125f, 0.693145751953125f), xc);
    r = __ffma2_rn(nn, make_float2(1.42860677e-06f, 1.42860677e-06f), r);
    float2 p = make_float2(1.0f / 5040.0f, 1.0f / 5040.0f);
    p = __ffma2_rn(p, r, make_float2(1.0f / 720.0f, 1.0f / 720.0f));
    p = __ffma2_rn(p, r, make_float2(1.0f / 120.0f, 1.0f / 120.0f));
    p = __ffma2_rn(p, r, make_float2(1.0f / 24.0f, 1.0f / 24.0f));
    p = __ffma2_rn(p, r, make_float2(1.0f / 6.0f, 1.0f / 6.0f));
    p = __ffma2_rn(p, r, make_float2(0.5f, 0.5f));
    p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
    p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
    const float2 two_n = make_float2(__int_as_float((static_cast<int>(n.x) + 127) << 23),
                                     __int_as_float((static_cast<int>(n.y) + 127) << 23));
    float2 e = __fmul2_rn(p, two_n);
    const float inf = __int_as_float(0x7f800000);
    if (x.x > 88.0f) e.x = inf;
    if (x.x < -87.0f) e.x = 0.0f;
    if (x.y > 88.0f) e.y = inf;
    if (x.y < -87.0f) e.y = 0.0f;
    return e;
}

// The two steps of h = SiLU(g) * u = g / (1 + e^-g) * u for two pairs of
// BF16-valued g and u (before the final rounding), one IEEE rounding per
// operation: the denominator 1 + e^-g, then the quotient times u.
__device__ __forceinline__ float2 silu_denom2(float2 g) {
    return __fadd2_rn(make_float2(1.0f, 1.0f), exp_cw2(make_float2(-g.x, -g.y)));
}

__device__ __forceinline__ float2 silu_mul2_from_denom(float2 g, float2 d, float2 u) {
    return __fmul2_rn(make_float2(__fdiv_rn(g.x, d.x), __fdiv_rn(g.y, d.y)), u);
}

__device__ __forceinline__ float2 silu_mul2_f32(float2 g, float2 u) {
    return silu_mul2_from_denom(g, silu_denom2(g), u);
}

// Test kernel: h[i] = bf16(SiLU(g[i]) * u[i]) on BF16 bit patterns, two
// elements per evaluation as in the GEMM epilogue (an odd last element is
// paired with itself).
__global__ void silu_mul_kernel(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* h) {
    const int64_t pairs = (n + 1) / 2;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < pairs;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t a = 2 * i, b = a + 1 < n ? a + 1 : a;
        const float2 v = silu_mul2_f32(make_float2(__uint_as_float(static_cast<uint32_t>(g[a]) << 16),
                                                   __uint_as_float(static_cast<uint32_t>(g[b]) << 16)),
                                       make_float2(__uint_as_float(static_cast<uint32_t>(u[a]) << 16),
                                                   __uint_as_float(static_cast<uint32_t>(u[b]) << 16)));
        const uint32_t w = f32x2_to_bf16x2(v.x, v.y);
        h[a] = static_cast<uint16_t>(w & 0xFFFFu);
        if (b != a) h[b] = static_cast<uint16_t>(w >> 16);
    }
}

}  // namespace fp8bs
