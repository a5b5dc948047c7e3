/*
 * fp8bs_oracle.c -- plain, slow, single-threaded CPU oracle for the FP8
 * fine-grained block-quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * What it restates.  The pages say that the main Transformer linear-layer
 * GEMMs run in blockwise FP8, following DeepSeek-V3's fine-grained block
 * quantization, while numerically sensitive operations and the training
 * state stay in BF16/FP32:
 *   - "Puro-2B: 普通实验室也能做预训练？" (training.farm blog), section
 *     "FP8：加快 RTX 5090 上的训练";
 *   - "Puro-2B: Poor Lab's Qwen2-1.5B Trained on RTX 5090 within $5090",
 *     part 1/7, section 2.1 "Pipeline at a Glance" and section 1 item 2;
 *   - bit.fan news article on Puro-2B, section "FP8 training and its trade-off".
 * The pages print none of the scheme's parameters.  The oracle takes the
 * published DeepSeek-V3 form of that scheme: 1x128 activation tiles,
 * 128x128 weight blocks, an FP32 scale s = amax/448 per tile, OCP E4M3FN
 * payloads, and FP32 promotion of the tensor-core partial sum once per
 * 128-wide K block.  Readings of the points the pages leave open are marked
 * "Reading:" below.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fPIC -shared (no FMA
 * contraction, so every product and sum rounds exactly where it is written).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* BF16 -> FP32: the BF16 bits are the top half of an FP32 word (exact). */
float orc_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* FP32 -> BF16, round to nearest, ties to even (finite inputs).  NaN is
 * kept quiet. */
uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lower = u & 0xffffu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* OCP FP8 E4M3FN decode: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 holds subnormals m * 2^-9; S.1111.111 is NaN; there
 * is no infinity; the largest finite value is S.1111.110 = 448. */
double orc_e4m3_decode(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int m = c & 7;
    double v;
    if (e == 0xf && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(8.0 + (double)m, e - 7 - 3);
    return sign ? -v : v;
}

/* FP32 -> OCP FP8 E4M3FN, round to nearest with ties to even, saturating
 * to the largest finite magnitude (448) instead of producing NaN.
 * Reading: the sign of zero is kept, so a negative value that rounds to
 * zero encodes as 0x80.  NaN encodes as 0x7F with its sign; +-Inf
 * saturates like any other value above 448. */
uint8_t orc_e4m3_encode(float v) {
    uint32_t u;
    memcpy(&u, &v, 4);
    uint8_t sign = (uint8_t)((u >> 31) << 7);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return (uint8_t)(sign | 0x7f); /* NaN */
    float x;
    memcpy(&x, &a, 4);                                 /* x = |v| */
    if (x >= 448.0f) return (uint8_t)(sign | 0x7e);    /* saturate */

    if (x >= 0.015625f) {
        /* Normal E4M3 range [2^-6, 448): x is a normal FP32 number.  Keep
         * the top 3 of its 23 mantissa bits and round the 20 dropped bits
         * to nearest, ties to even.  A carry out of the mantissa moves into
         * the exponent field, which is the right result. */
        int e = (int)(a >> 23) - 127; /* -6 .. 8 */
        uint32_t mant = a & 0x7fffffu;
        uint32_t keep = mant >> 20;
        uint32_t rest = mant & 0xfffffu;
        uint32_t code = ((uint32_t)(e + 7) << 3) | keep;
        if (rest > 0x80000u || (rest == 0x80000u && (keep & 1u))) code += 1u;
        if (code > 0x7eu) code = 0x7eu; /* 464 <= x < 448+32 rounds past 448 */
        return (uint8_t)(sign | code);
    }

    /* Subnormal E4M3 range: the representable values are m * 2^-9 for
     * m = 0..7 (m = 8 is 2^-6, code 0x08).  y = x * 512 is exact; round it
     * to the nearest integer, ties to even. */
    {
        float y = x * 512.0f;
        uint32_t m = (uint32_t)y;   /* floor, y < 8 */
        float frac = y - (float)m;  /* exact */
        if (frac > 0.5f || (frac == 0.5f && (m & 1u))) m += 1u;
        return (uint8_t)(sign | m);
    }
}

/* ------------------------------------------------------------------ */
/* Per-tile scale                                                      */
/* ------------------------------------------------------------------ */

/* Scale and its reciprocal multiplier for one tile with absolute maximum
 * amax (DeepSeek-V3 form: the tile's largest magnitude maps to E4M3's 448).
 *   s   = amax / 448     (FP32 division, round to nearest) -- stored
 *   inv = 448 / amax     (FP32 division, round to nearest) -- applied
 * Reading (payload form): the payload is encode(x * inv) with one rounded
 * FP32 multiply, not encode(x / s).
 * Reading (all-zero tile): amax == 0 gives s = 1 and inv = 1, so every
 * payload is a signed zero.
 * Reading (tiny tiles): when 448/amax overflows FP32 it is clamped to
 * FLT_MAX, so zeros stay zero instead of becoming 0*Inf = NaN. */
static void tile_scale(float amax, float* s, float* inv) {
    if (amax == 0.0f) {
        *s = 1.0f;
        *inv = 1.0f;
        return;
    }
    /* The volatile copy keeps GCC 13's floating-point range propagation from
     * folding amax/448 to 0 on the branch where 448/amax overflows (there
     * the quotient is a nonzero subnormal, not 0). */
    volatile float va = amax;
    *s = va / 448.0f;
    float r = 448.0f / va;
    if (r > FLT_MAX) r = FLT_MAX;
    *inv = r;
}

/* ------------------------------------------------------------------ */
/* Quantizers                                                          */
/* ------------------------------------------------------------------ */

/* Token count rounded up to whole 128-token blocks.  Reading (token
 * tails): when the number of tokens is not a multiple of 128, token-major
 * arrays -- row scales, the transposed payload and its scales -- keep a
 * leading dimension of Mp = this many tokens; the padding tokens count as
 * zeros (payload 0x00, and a padding-only tile is an all-zero tile, s = 1). */
static int64_t padded_tokens(int64_t rows) { return (rows + 127) / 128 * 128; }

/* 1x128 row-wise activation quantization.
 * x: BF16 [rows][cols]; q: E4M3 [rows][cols]; s: FP32 [cols/128][Mp]
 * (scale of tile (r, b) at s[b*Mp + r]; rows r >= `rows` hold the all-zero
 * tile scale 1).  cols % 128 == 0; rows > 0. */
void orc_quant_rowwise_1x128(const uint16_t* x, int64_t rows, int64_t cols,
                             uint8_t* q, float* s) {
    int64_t nb = cols / 128, mp = padded_tokens(rows);
    for (int64_t r = 0; r < mp; r++) {
        for (int64_t b = 0; b < nb; b++) {
            if (r >= rows) {
                s[b * mp + r] = 1.0f;
                continue;
            }
            const uint16_t* t = x + r * cols + b * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; i++) {
                float a = fabsf(orc_bf16_to_f32(t[i]));
                if (a > amax) amax = a;
            }
            float sc, inv;
            tile_scale(amax, &sc, &inv);
            s[b * mp + r] = sc;
            for (int i = 0; i < 128; i++)
                q[r * cols + b * 128 + i] = orc_e4m3_encode(orc_bf16_to_f32(t[i]) * inv);
        }
    }
}

/* 128x1 token-dim quantization, written transposed (for the weight
 * gradient, which contracts over tokens).
 * x: BF16 [rows][cols]; qT: E4M3 [cols][Mp]; sT: FP32 [Mp/128][cols]
 * (scale of the tile (column c, token block b) at sT[b*cols + c]).
 * Reading: the transposed operand is quantized from the original BF16
 * tensor, not requantized from its 1x128 FP8 form.  The last token block
 * may hold fewer than 128 tokens: its amax is taken over the tokens present
 * and the padding tokens' payload is 0x00 (see padded_tokens). */
void orc_quant_colwise_128x1_T(const uint16_t* x, int64_t rows, int64_t cols,
                               uint8_t* qT, float* sT) {
    int64_t mp = padded_tokens(rows), nb = mp / 128;
    for (int64_t c = 0; c < cols; c++) {
        for (int64_t b = 0; b < nb; b++) {
            int64_t n = rows - b * 128;
            if (n > 128) n = 128;
            float amax = 0.0f;
            for (int64_t i = 0; i < n; i++) {
                float a = fabsf(orc_bf16_to_f32(x[(b * 128 + i) * cols + c]));
                if (a > amax) amax = a;
            }
            float sc, inv;
            tile_scale(amax, &sc, &inv);
            sT[b * cols + c] = sc;
            for (int64_t i = 0; i < 128; i++)
                qT[c * mp + b * 128 + i] =
                    i < n ? orc_e4m3_encode(orc_bf16_to_f32(x[(b * 128 + i) * cols + c]) * inv) : 0x00;
        }
    }
}

/* 128x128 block weight quantization.
 * w: BF16 [n][k]; q: E4M3 [n][k]; qT: E4M3 [k][n] (the same bytes,
 * transposed; may be NULL); s: FP32 [n/128][k/128]. */
void orc_quant_weight_128x128(const uint16_t* w, int64_t n, int64_t k,
                              uint8_t* q, uint8_t* qT, float* s) {
    int64_t nbn = n / 128, nbk = k / 128;
    for (int64_t bn = 0; bn < nbn; bn++) {
        for (int64_t bk = 0; bk < nbk; bk++) {
            float amax = 0.0f;
            for (int i = 0; i < 128; i++)
                for (int j = 0; j < 128; j++) {
                    float a = fabsf(orc_bf16_to_f32(w[(bn * 128 + i) * k + bk * 128 + j]));
                    if (a > amax) amax = a;
                }
            float sc, inv;
            tile_scale(amax, &sc, &inv);
            s[bn * nbk + bk] = sc;
            for (int i = 0; i < 128; i++)
                for (int j = 0; j < 128; j++) {
                    int64_t r = bn * 128 + i, c = bk * 128 + j;
                    uint8_t code = orc_e4m3_encode(orc_bf16_to_f32(w[r * k + c]) * inv);
                    q[r * k + c] = code;
                    if (qT) qT[c * n + r] = code;
                }
        }
    }
}

/* ------------------------------------------------------------------ */
/* GEMMs with per-128-K promotion                                      */
/* ------------------------------------------------------------------ */

/* Decoded value of every E4M3 code, filled when the library is loaded (so
 * concurrent callers on several threads only ever read it). */
static double g_dec[256];

__attribute__((constructor)) static void dec_table_init(void) {
    for (int c = 0; c < 256; c++) g_dec[c] = orc_e4m3_decode((uint8_t)c);
}

/* One output element of a block-scaled product.
 *   a, b  : the two E4M3 rows being contracted (length kc, kc % 128 == 0)
 *   sa[j] : FP32 scale of a's j-th 128-block (stride sa_stride)
 *   sb[j] : FP32 scale of b's j-th 128-block (stride sb_stride)
 * For each 128-block j in increasing order:
 *   P_j = sum of the 128 products of decoded payloads, exact in double
 *         (every product is a multiple of 2^-18 below 2^17.6, so any sum
 *         of 128 of them fits in 43 significant bits);
 *   acc = fmaf((float)P_j, sa_j * sb_j, acc)   (FP32; sa_j*sb_j rounded)
 * Reading: promotion uses one fused multiply-add per block, starting from
 * acc = 0.  Also returns sum_k |a_k b_k| of the dequantized values. */
static float block_dot(const uint8_t* a, const uint8_t* b, int64_t kc,
                       const float* sa, int64_t sa_stride,
                       const float* sb, int64_t sb_stride, double* sumabs) {
    float acc = 0.0f;
    double sab_total = 0.0;
    for (int64_t j = 0; j < kc / 128; j++) {
        double p = 0.0, pabs = 0.0;
        for (int i = 0; i < 128; i++) {
            double t = g_dec[a[j * 128 + i]] * g_dec[b[j * 128 + i]];
            p += t;
            pabs += fabs(t);
        }
        float scale = sa[j * sa_stride] * sb[j * sb_stride];
        acc = fmaf((float)p, scale, acc);
        sab_total += pabs * (double)sa[j * sa_stride] * (double)sb[j * sb_stride];
    }
    *sumabs = sab_total;
    return acc;
}

static void emit(float acc, double sabs, int64_t idx, float* out_f32,
                 uint16_t* out_bf16, double* out_sumabs) {
    if (out_f32) out_f32[idx] = acc;
    if (out_bf16) out_bf16[idx] = orc_f32_to_bf16(acc);
    if (out_sumabs) out_sumabs[idx] = sabs;
}

/* fprop: Y[m][n] = sum_b sX[b][m] * sW[n/128][b] * P_b[m][n],
 *        P_b[m][n] = sum_{k in block b} Xq[m][k] * Wq[n][k].
 * Xq [M][K], sX [K/128][ldsx] (ldsx >= M; the quantizer writes
 * Mp = M rounded up to 128 tokens), Wq [N][K], sW [N/128][K/128].
 * Computes the rows listed in `rows` (nrows of them); output row i is
 * written at out[i*N .. i*N+N).  Any output pointer may be NULL. */
void orc_gemm_fprop(const uint8_t* xq, const float* sx, const uint8_t* wq,
                    const float* sw, int64_t M, int64_t N, int64_t K, int64_t ldsx,
                    const int64_t* rows, int64_t nrows, float* out_f32,
                    uint16_t* out_bf16, double* out_sumabs) {
    int64_t kb = K / 128;
    for (int64_t i = 0; i < nrows; i++) {
        int64_t m = rows[i];
        for (int64_t n = 0; n < N; n++) {
            double sabs;
            float acc = block_dot(xq + m * K, wq + n * K, K, sx + m, ldsx,
                                  sw + (n / 128) * kb, 1, &sabs);
            emit(acc, sabs, i * N + n, out_f32, out_bf16, out_sumabs);
        }
    }
}

/* dgrad: dX[m][k] = sum_b sdY[b][m] * sW[b][k/128] * P_b[m][k],
 *        P_b[m][k] = sum_{n in block b} dYq[m][n] * Wq[n][k].
 * dYq [M][N], sdY [N/128][ldsdy], Wq [N][K] (the forward payload: the oracle
 * reads the weight in its own layout), sW [N/128][K/128].  Output rows as
 * for fprop, each of length K. */
void orc_gemm_dgrad(const uint8_t* dyq, const float* sdy, const uint8_t* wq,
                    const float* sw, int64_t M, int64_t N, int64_t K, int64_t ldsdy,
                    const int64_t* rows, int64_t nrows, float* out_f32,
                    uint16_t* out_bf16, double* out_sumabs) {
    int64_t kb = K / 128;
    uint8_t col[65536];
    if (N > 65536) return;
    for (int64_t k = 0; k < K; k++) {
        for (int64_t n = 0; n < N; n++) col[n] = wq[n * K + k]; /* column k of W */
        for (int64_t i = 0; i < nrows; i++) {
            int64_t m = rows[i];
            double sabs;
            float acc = block_dot(dyq + m * N, col, N, sdy + m, ldsdy,
                                  sw + k / 128, kb, &sabs);
            emit(acc, sabs, i * K + k, out_f32, out_bf16, out_sumabs);
        }
    }
}

/* wgrad: dW[n][k] = sum_b sdYT[b][n] * sXT[b][k] * P_b[n][k],
 *        P_b[n][k] = sum_{m in block b} dYTq[n][m] * XTq[k][m].
 * dYTq [N][M], sdYT [M/128][N], XTq [K][M], sXT [M/128][K], where M is
 * the padded token count (the transposed quantizer's padding tokens are
 * zeros and add nothing).  The rows listed are output rows n; output row i
 * has length K. */
void orc_gemm_wgrad(const uint8_t* dytq, const float* sdyt, const uint8_t* xtq,
                    const float* sxt, int64_t M, int64_t N, int64_t K,
                    const int64_t* rows, int64_t nrows, float* out_f32,
                    uint16_t* out_bf16, double* out_sumabs) {
    for (int64_t i = 0; i < nrows; i++) {
        int64_t n = rows[i];
        for (int64_t k = 0; k < K; k++) {
            double sabs;
            float acc = block_dot(dytq + n * M, xtq + k * M, M, sdyt + n, N,
                                  sxt + k, K, &sabs);
            emit(acc, sabs, i * K + k, out_f32, out_bf16, out_sumabs);
        }
    }
}

/* Bulk encoder used by the tests to sweep FP32 bit patterns. */
void orc_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = orc_e4m3_encode(v[i]);
}

/* Bulk encoder over a contiguous range of FP32 bit patterns
 * [first, first+n). */
void orc_e4m3_encode_bits(uint32_t first, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; i++) {
        uint32_t u = first + (uint32_t)i;
        float f;
        memcpy(&f, &u, 4);
        out[i] = orc_e4m3_encode(f);
    }
}

void orc_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
    for (int64_t i = 0; i < n; i++) out[i] = orc_e4m3_decode(c[i]);
}

/* ------------------------------------------------------------------ */
/* SwiGLU activation between the gate+up and down projections          */
/* ------------------------------------------------------------------ */

/* e^x in FP32 by the Cody-Waite method (W. J. Cody and W. Waite, "Software
 * Manual for the Elementary Functions", 1980): x = n ln2 + r with
 * n = rint(x log2 e) and r computed with a two-part ln 2 (the high part
 * has 16 significant bits, so n * LN2_HI is exact for |n| < 256), then
 * e^r by its Taylor polynomial of degree 7 (|r| <= ln2/2, remainder below
 * 2^-27 relative), then the factor 2^n.  Every step is one IEEE FP32
 * operation in the order written (fmaf where written, no contraction).
 * Reading (range): x > 88 gives +Inf and x < -87 gives 0, so 2^n stays a
 * normal power of two; the activation's inputs lie far inside. */
static const float LOG2E_F = 1.44269502f;          /* log2(e) rounded to FP32 */
static const float LN2_HI_F = 0.693145751953125f;  /* 45426 / 2^16 */
static const float LN2_LO_F = 1.42860677e-06f;     /* ln 2 - LN2_HI, rounded */

float orc_exp_cw(float x) {
    if (x > 88.0f) return INFINITY;
    if (x < -87.0f) return 0.0f;
    float n = rintf(x * LOG2E_F);
    float r = fmaf(-n, LN2_HI_F, x);
    r = fmaf(-n, LN2_LO_F, r);
    float p = 1.0f / 5040.0f;
    p = fmaf(p, r, 1.0f / 720.0f);
    p = fmaf(p, r, 1.0f / 120.0f);
    p = fmaf(p, r, 1.0f / 24.0f);
    p = fmaf(p, r, 1.0f / 6.0f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    uint32_t bits = (uint32_t)((int32_t)n + 127) << 23; /* 2^n, n in [-126, 127] */
    float two_n;
    memcpy(&two_n, &bits, 4);
    return p * two_n;
}

/* h = SiLU(g) * u of one element, SiLU(g) = g / (1 + e^-g): g and u are
 * the BF16 outputs of the gate and up projections (what a BF16 forward
 * product holds); the activation runs in FP32 and h is rounded to BF16.
 * Reading: the pages keep the activation out of the FP8 path and give no
 * formula; this is the SwiGLU form, g * sigmoid(g) * u, evaluated as
 * g / (1 + e^-g) * u with one rounding per operation. */
uint16_t orc_silu_mul_bf16(uint16_t g_bits, uint16_t u_bits) {
    float g = orc_bf16_to_f32(g_bits);
    float u = orc_bf16_to_f32(u_bits);
    float t = orc_exp_cw(-g);
    float d = 1.0f + t;
    float sg = g / d;
    return orc_f32_to_bf16(sg * u);
}

void orc_silu_mul_array(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* h) {
    for (int64_t i = 0; i < n; i++) h[i] = orc_silu_mul_bf16(g[i], u[i]);
}

void orc_exp_cw_array(const float* x, int64_t n, float* out) {
    for (int64_t i = 0; i < n; i++) out[i] = orc_exp_cw(x[i]);
}
