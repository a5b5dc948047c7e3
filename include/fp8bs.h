/*
 * fp8bs.h -- C ABI of the FP8 fine-grained block-quantized linear layer for
 * NVIDIA B300 (sm_103a).
 *
 * The method.  The Puro-2B pages put the main Transformer linear-layer GEMMs
 * on a blockwise FP8 path that follows DeepSeek-V3's fine-grained block
 * quantization, and keep numerically sensitive operations and the training
 * state in BF16/FP32 ("Puro-2B: 普通实验室也能做预训练？", section
 * "FP8：加快 RTX 5090 上的训练"; "Puro-2B: Poor Lab's Qwen2-1.5B Trained on
 * RTX 5090 within $5090", part 1/7, section 2.1 and section 1 item 2; bit.fan
 * news article, section "FP8 training and its trade-off").  The pages print
 * none of the scheme's parameters; this library implements its published
 * DeepSeek-V3 form:
 *   - activations: one FP32 scale per 1x128 tile (a row segment of 128
 *     elements along the contraction dimension);
 *   - weights: one FP32 scale per 128x128 block;
 *   - scale s = amax / 448 (FP32 division); payload q = E4M3(x * (448/amax))
 *     with one rounded FP32 multiply, round-to-nearest-even, saturating at
 *     +-448 (OCP E4M3FN); an all-zero tile stores s = 1; when 448/amax
 *     overflows FP32 the multiplier is clamped to FLT_MAX;
 *   - GEMMs: each 128-wide K block's partial sum P_b comes from the tensor
 *     cores in FP32 and is promoted outside them:
 *     acc = fma(P_b, sa_b * sb_b, acc), then the output is rounded to BF16;
 *   - weight gradient: X and dY are requantized along the token dimension
 *     (128x1 tiles) from their BF16 originals and stored transposed, so the
 *     token dimension becomes the contraction dimension.
 *
 * Library state: a per-device status word, per-device split-K scratch
 * registration, and a cache of encoded TMA tensor maps (keyed by pointer
 * and shape; an entry is exactly what re-encoding would produce).
 *
 * Conventions for every entry point:
 *   - All tensors are row-major and contiguous; "[a][b]" means a rows of b.
 *   - All data pointers are DEVICE pointers (cudaMalloc / PyTorch CUDA
 *     memory) on the current device, 16-byte aligned.  The caller owns every
 *     buffer; the library never allocates or frees per call.
 *   - Feature dimensions (K, N, and both dimensions of a weight) must be
 *     positive multiples of 128.  The token count (M, the rows of X, dY, Y,
 *     dX) may be any positive number: token-major arrays -- row scales,
 *     transposed payloads and their scales -- then have a leading dimension
 *     of Mp = M rounded up to a multiple of 128.  The last 128x1 token tile
 *     covers the tokens present; padding tokens are stored as zero payloads
 *     (and padding rows' scales as 1), so they add nothing to a product.
 *     Everything else is laid out exactly as for M = Mp.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous and stream-ordered; the host never synchronizes.
 *   - Argument errors return a status and launch nothing.  Errors that
 *     happen on the device (a bounded wait that expired) are recorded in a
 *     per-device status word read by fp8bs_get_device_status().
 *   - Outputs are bitwise deterministic (no atomics, fixed reduction order).
 *   - Calls on different streams are thread-safe; output buffers of calls
 *     that may overlap in time must not alias.
 */
#ifndef FP8BS_H_
#define FP8BS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fp8bs_status {
    FP8BS_OK = 0,
    FP8BS_ERR_INVALID_ARG = 1, /* a required pointer is NULL, or bad flags */
    FP8BS_ERR_SHAPE = 2,       /* a dimension is <= 0, not a multiple of 128, or too large */
    FP8BS_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
    FP8BS_ERR_ARCH = 4,        /* no CUDA device, or the current device is not compute capability 10.3 (sm_103) */
    FP8BS_ERR_LAUNCH = 5,      /* the CUDA runtime reported an error at launch */
    FP8BS_ERR_TIMEOUT = 6,     /* a bounded wait inside a kernel expired (device status) */
    FP8BS_ERR_CUDA = 7         /* a CUDA runtime call failed (device status query) */
} fp8bs_status;

/* Layout flags for fp8bs_quantize_act (may be OR-ed: one read of x then
 * writes both layouts). */
#define FP8BS_ROWWISE 1u   /* 1x128 tiles: q [rows][cols], s [cols/128][rows] */
#define FP8BS_COLWISE_T 2u /* 128x1 tiles, transposed: qT [cols][rows], sT [rows/128][cols] */

/*
 * Activation (or activation-gradient) quantization.
 *   x      : BF16 [rows][cols], read only.
 *   flags  : FP8BS_ROWWISE and/or FP8BS_COLWISE_T (at least one).
 *   q, s   : with FP8BS_ROWWISE -- E4M3 payload [rows][cols] and FP32
 *            scales [cols/128][Mp]: the scale of the tile holding
 *            x[r][128b .. 128b+127] is s[b*Mp + r] (Mp: rows rounded up to
 *            128; s is 1 for r >= rows).  Scales are stored
 *            k-block-major so that the 128 row scales of one GEMM tile are
 *            contiguous.  Ignored (may be NULL) without the flag.
 *   qT, sT : with FP8BS_COLWISE_T -- the 128x1-tiled payload written
 *            transposed, qT [cols][Mp] (qT[c][r] encodes x[r][c]; 0 for
 *            r >= rows), and FP32 scales sT [Mp/128][cols]: the scale of the
 *            tile holding x[128b .. 128b+127][c] (the tokens present) is
 *            sT[b*cols + c].  Ignored (may be NULL)
 *            without the flag.
 * rows is the token count M for X or dY; cols is K (for X) or N (for dY).
 * Passage: the pages' fine-grained (tile-wise) activation quantization,
 * "FP8：加快 RTX 5090 上的训练" and section 2.1 of the arXiv text.
 */
int fp8bs_quantize_act(const void* x, int64_t rows, int64_t cols, unsigned flags,
                       uint8_t* q, float* s, uint8_t* qT, float* sT, void* stream);

/*
 * Weight quantization with 128x128 blocks.
 *   w  : BF16 [n][k] (out features x in features), read only.
 *   q  : E4M3 payload [n][k] (used by fprop).
 *   qT : NULL, or E4M3 [k][n] holding the same bytes transposed (used by
 *        dgrad, which contracts over n).  A 128x128 block's scale is the
 *        same in both layouts.
 *   s  : FP32 [n/128][k/128]; block (i, j) covers w[128i..][128j..].
 * Passage: the pages' block-wise weight quantization (same sections).
 */
int fp8bs_quantize_weight(const void* w, int64_t n, int64_t k, uint8_t* q, uint8_t* qT,
                          float* s, void* stream);

/*
 * Forward GEMM  Y = X W^T  (BF16 out [M][N]).
 *   xq [M][K] E4M3 with sx [K/128][Mp] (from fp8bs_quantize_act, ROWWISE),
 *   wq [N][K] E4M3 with sw [N/128][K/128] (from fp8bs_quantize_weight).
 *   Y[m][n] = bf16( sum_b fma-chain of P_b[m][n] * (sx[b][m] * sw[n/128][b]) )
 *   with P_b the FP32 tensor-core sum over k in [128b, 128b+128).
 * Passage: "main linear-layer GEMMs on the FP8 path" (blog section
 * "FP8：加快 RTX 5090 上的训练"; arXiv part 1/7, section 2.1).
 */
int fp8bs_gemm_fprop(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw,
                     void* y, int64_t M, int64_t N, int64_t K, void* stream);

/*
 * Forward GEMM with an FP8 output for the next linear:  Y = X W^T, then Y's
 * 1x128 row-wise quantization, in the GEMM's epilogue (no extra pass over Y).
 *   xq, sx, wq, sw, M, N, K : as for fp8bs_gemm_fprop.
 *   y  : BF16 [M][N] output, or NULL to skip it.
 *   yq : E4M3 [M][N] and sy : FP32 [N/128][Mp] (Mp = M rounded up to 128;
 *        padding rows get s = 1) -- exactly what fp8bs_quantize_act with
 *        FP8BS_ROWWISE writes for the BF16 Y: each 1x128 tile of the
 *        BF16-rounded product gets s = amax/448 and E4M3(y * 448/amax).
 * The weight gradient of the next linear still needs Y's 128x1 transposed
 * quantization (fp8bs_quantize_act with FP8BS_COLWISE_T on the BF16 Y).
 * Passage: the pages keep the FP8 path on the main linear GEMMs and their
 * inputs (blog section "FP8：加快 RTX 5090 上的训练"); this fuses the
 * quantization of a linear's FP8 input into the producing GEMM.
 */
int fp8bs_gemm_fprop_quant(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw, void* y,
                           uint8_t* yq, float* sy, int64_t M, int64_t N, int64_t K, void* stream);

/*
 * Gate+up forward GEMM with the SwiGLU activation and the down projection's
 * FP8 input computed in the epilogue:
 *   H = SiLU(G) * U,  G = X Wg^T, U = X Wu^T  (BF16-rounded, as fprop gives),
 *   SiLU(g) = g / (1 + e^-g) in FP32, H rounded to BF16, then H's 1x128
 *   row-wise quantization.
 *   xq, sx : X as for fp8bs_gemm_fprop ([M][K], [K/128][Mp]).
 *   wq, sw : the quantized gate+up weight [N2][K] (N2 = 2 I, a multiple of
 *            256) whose rows alternate in 128-row blocks: rows 256j..256j+127
 *            are gate rows 128j..128j+127, rows 256j+128..256j+255 the up rows
 *            of the same outputs (fp8bs_quantize_weight on that interleaved W
 *            gives wq, sw [N2/128][K/128]).
 *   h      : BF16 [M][I] output, or NULL to skip it.
 *   hq, sh : E4M3 [M][I] and FP32 [I/128][Mp] -- what fp8bs_quantize_act
 *            with FP8BS_ROWWISE writes for H.
 * e^x is computed by Cody-Waite reduction with a degree-7 Taylor polynomial
 * (one IEEE operation per step), so every H is a fixed function of G and U;
 * fp8bs_debug_silu_mul runs the same activation on arrays.
 * Passage: the activation stays out of the FP8 path (blog section
 * "FP8：加快 RTX 5090 上的训练"); its output is the down projection's FP8
 * input, quantized here without a pass over H.
 */
int fp8bs_gemm_fprop_swiglu_quant(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw, void* h,
                                  uint8_t* hq, float* sh, int64_t M, int64_t N2, int64_t K, void* stream);

/*
 * Data-gradient GEMM  dX = dY W  (BF16 out [M][K]); contraction over N.
 *   dyq [M][N] E4M3 with sdy [N/128][Mp] (fp8bs_quantize_act on dY, ROWWISE),
 *   wqT [K][N] E4M3 (the transposed payload from fp8bs_quantize_weight),
 *   sw  [N/128][K/128] (the same weight scales as fprop; block (b, k/128)
 *       scales contraction block b of output column k).
 * Passage: as for fprop (the backward linear GEMMs are on the FP8 path).
 */
int fp8bs_gemm_dgrad(const uint8_t* dyq, const float* sdy, const uint8_t* wqT, const float* sw,
                     void* dx, int64_t M, int64_t N, int64_t K, void* stream);

/*
 * Weight-gradient GEMM  dW = dY^T X  (BF16 out [N][K]); contraction over
 * the M tokens.
 *   dyTq [N][Mp] E4M3 with sdyT [Mp/128][N] (fp8bs_quantize_act on dY,
 *        COLWISE_T), xTq [K][Mp] E4M3 with sxT [Mp/128][K] (the same on X);
 *        M is the token count (the padding tokens contribute zero).
 *   dW[n][k] = bf16( fma-chain over token blocks b of
 *              P_b[n][k] * (sdyT[b][n] * sxT[b][k]) ).
 * With a registered scratch buffer (fp8bs_set_workspace) the contraction
 * may be split across CTAs; see there.
 * Passage: as for fprop.
 */
int fp8bs_gemm_wgrad(const uint8_t* dyTq, const float* sdyT, const uint8_t* xTq, const float* sxT,
                     void* dw, int64_t M, int64_t N, int64_t K, void* stream);

/*
 * Weight gradient accumulated in FP32:  dW += dY^T X.
 *   Same operands, layouts and promotion as fp8bs_gemm_wgrad, but dw is an
 *   FP32 [N][K] buffer that the result is added to (TMA reduce-add: each
 *   element receives one FP32 add, in stream order across calls), with no
 *   BF16 rounding: for gradient accumulation over micro-batches in the
 *   master-gradient precision that the training state keeps (the pages keep
 *   master weights and optimizer state in FP32/BF16).  Uses the split-K
 *   scratch like fp8bs_gemm_wgrad.
 * Passage: as for fprop; "numerically sensitive operations and persistent
 * training states ... in BF16 or FP32" (arXiv part 1/7, section 2.1).
 */
int fp8bs_gemm_wgrad_accumulate_f32(const uint8_t* dyTq, const float* sdyT, const uint8_t* xTq, const float* sxT,
                                    float* dw, int64_t M, int64_t N, int64_t K, void* stream);

/* Product codes of fp8bs_gemm_group and fp8bs_gemm_workspace_bytes. */
#define FP8BS_OP_FPROP 0
#define FP8BS_OP_DGRAD 1
#define FP8BS_OP_WGRAD 2

/*
 * Several products in one persistent launch (grouped GEMM).
 *
 * A decoder layer's linears give independent products of the same kind in
 * each phase of a step -- the forward products of its four linears, their
 * data gradients, their weight gradients.  Launched one by one, each ends
 * with a partly idle last wave of its 128 x 256 tiles; grouped, the tiles of
 * all members are dealt to the persistent CTAs as one list (member 0's tiles
 * first), so only the group's last wave is ragged.
 *   gemms[count] : 1 <= count <= FP8BS_GROUP_MAX products, each given by its
 *                  op (FP8BS_OP_FPROP, _DGRAD or _WGRAD) and exactly the
 *                  arguments of that op's entry point (a = xq / dyq / dyTq,
 *                  sa = sx / sdy / sdyT, b = wq / wqT / xTq, sb = sw / sw /
 *                  sxT, out = y / dx / dw as BF16).  Forward and data-gradient
 *                  products may share a group; weight gradients form groups
 *                  of their own (their promotion differs).
 * With registered scratch (fp8bs_set_workspace) large enough for every
 * member's split plan, each member splits as its own entry point would, in
 * its own region of the scratch (regions in member order; a member that no
 * longer fits stays whole), and each output is bitwise equal to the
 * member's own call; without scratch, to its unsplit result.  Outputs must
 * not overlap each other or any input.  Errors: FP8BS_ERR_INVALID_ARG for a NULL array, a
 * count out of range, an unknown op or mixed weight-gradient and other
 * members; otherwise as for the members' entry points (checked before
 * anything is launched).
 */
#define FP8BS_GROUP_MAX 4
typedef struct fp8bs_gemm_args {
    int op;
    const uint8_t* a;
    const float* sa;
    const uint8_t* b;
    const float* sb;
    void* out;
    int64_t M, N, K;
} fp8bs_gemm_args;
int fp8bs_gemm_group(const fp8bs_gemm_args* gemms, int count, void* stream);

/*
 * Scratch memory for the GEMMs' split-K path (caller-owned).
 *
 * When the output tiles (128 x 256) of a product do not fill the last wave
 * of the 148 SMs well and the contraction is long enough to pay for moving
 * FP32 partial sums (a weight gradient over many tokens with few tiles, e.g.
 * 2048 x 5632 outputs), the contraction of the last wave's tiles, or of all
 * tiles, is split into 2-8 parts computed by different CTAs.  Each part
 * keeps the per-128-K promotion chain over its own K blocks and publishes
 * its FP32 partial sum; whichever part finishes last adds all of them in a
 * fixed order (part 0 + part 1 + ...), so results stay bitwise
 * deterministic, and no CTA ever waits for another (the parts need not be
 * resident at the same time).  Forward products with the SwiGLU epilogue
 * are not split.  The partial sums go through this scratch buffer:
 *
 *   fp8bs_gemm_workspace_bytes(op, M, N, K): bytes the current device needs
 *     for product `op` (FP8BS_OP_FPROP, _DGRAD, _WGRAD) with the arguments
 *     of that product's entry point; 0 if it would not split; a negative
 *     status on bad shapes, an unknown op or no usable device.
 *   fp8bs_gemm_wgrad_workspace_bytes(M, N, K): the same for FP8BS_OP_WGRAD.
 *   fp8bs_set_workspace(ws, bytes): registers `bytes` of DEVICE memory at
 *     `ws` (256-byte aligned, bytes >= 64 KiB; NULL and 0 unregister) as the
 *     current device's scratch.  The library zeroes its first 64 KiB (the
 *     arrival counters) with a blocking cudaMemset and keeps the pointer; the
 *     caller keeps the memory alive and unmodified while it is registered,
 *     and registers only while no GEMM is running.  Without a large enough
 *     registration a product simply does not split.  GEMMs that share one
 *     scratch must not overlap in time (two streams would race on it).
 */
int fp8bs_set_workspace(void* ws, int64_t bytes);
int64_t fp8bs_gemm_workspace_bytes(int op, int64_t M, int64_t N, int64_t K);
int64_t fp8bs_gemm_wgrad_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * Weight gradient for callers that cannot allocate.
 *
 * The paper has no counterpart of this call; it exists for library users.
 * fp8bs_gemm_wgrad needs scratch memory from its caller to split small
 * weight gradients (fp8bs_set_workspace).  Some callers cannot provide any:
 * code embedded in a host framework that owns all device memory through its
 * own pool and exposes no allocator to plug-ins, or latency-critical loops
 * in which a cudaMalloc (which can synchronize the whole device and take
 * arbitrarily long) is not acceptable.  This entry point computes the same
 * dW = dY^T X with the same arguments, layouts, split plan and results as
 * fp8bs_gemm_wgrad, but takes its scratch from a static device array of
 * FP8BS_NOALLOC_SCRATCH_BYTES (48 MiB) compiled into the library, which
 * every GPU that loads the library holds until the process exits.  Neither
 * the library nor the caller allocates anything: the caller passes only the
 * inputs and the output, as for fp8bs_gemm_wgrad.
 *
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call outside any stream
 *     capture.
 *   - Shapes whose split plan needs more scratch than the array holds are
 *     rejected with FP8BS_ERR_SHAPE before anything is launched
 *     (fp8bs_gemm_wgrad_workspace_bytes tells the need).
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents; each call tags its arrival counters with its own
 *     number, so nothing needs clearing first.  Two calls that may overlap
 *     on the GPU (different streams, no ordering between them) race on the
 *     array and give wrong results.
 *   - Errors as for fp8bs_gemm_wgrad; FP8BS_ERR_CUDA if the array's address
 *     cannot be looked up.
 */
#define FP8BS_NOALLOC_SCRATCH_BYTES (48ull << 20)
int fp8bs_gemm_wgrad_noalloc(const uint8_t* dyTq, const float* sdyT, const uint8_t* xTq, const float* sxT,
                             void* dw, int64_t M, int64_t N, int64_t K, void* stream);

/* Synchronizes `stream`, then returns and clears the current device's
 * status word: FP8BS_OK, FP8BS_ERR_TIMEOUT (a kernel gave up a bounded
 * wait and returned early; its outputs are undefined), or FP8BS_ERR_CUDA
 * if the synchronization itself failed. */
int fp8bs_get_device_status(void* stream);

/* Human-readable name of a status code (static storage). */
const char* fp8bs_status_string(int status);

/* Number of kernels launched by this process through the library (all
 * entry points, all devices); a diagnostic counter. */
int64_t fp8bs_launch_count(void);

/* Number of TMA tensor maps the library has encoded with the driver.  The
 * GEMM entry points keep encoded maps in a cache keyed by pointer, shape,
 * stride, box and swizzle (an encoded map depends on nothing else), so a
 * repeated call on the same buffers encodes none; a diagnostic counter. */
int64_t fp8bs_debug_tensor_map_encodes(void);

/*
 * Test hooks (not for production use).
 *   fp8bs_debug_set_wait_timeout_ns: the limit of every bounded device wait
 *     (default 2e9 ns); 0 restores the default.
 *   fp8bs_debug_force_tile_order: GEMM launches take their tiles in column
 *     strips `strip` tiles wide (capped at the output's tile columns; 1:
 *     column by column) instead of the order fp8bs_debug_tile_order would
 *     choose, until reset with 0.  Outputs do not depend on the order except
 *     through which tiles a split plan splits (the split tiles are the last
 *     ones in that order).  FP8BS_ERR_INVALID_ARG for a negative width.
 *   fp8bs_debug_set_fault: when 1, the next GEMM launch withholds one
 *     operand copy so that the kernel's bounded wait expires and it reports
 *     FP8BS_ERR_TIMEOUT without faulting; reset to 0 after that launch.
 *   fp8bs_debug_e4m3_encode_bits: runs the kernels' FP32->E4M3 encoder on
 *     the FP32 values whose bit patterns are first .. first+n-1, writing n
 *     codes to the device buffer `out`.
 *   fp8bs_debug_silu_mul: h[i] = bf16(SiLU(g[i]) * u[i]) on BF16 bit patterns
 *     (device arrays of n elements), the activation of
 *     fp8bs_gemm_fprop_swiglu_quant.
 *   fp8bs_debug_set_flags: test modes of the GEMMs, until reset with 0.
 *     FP8BS_DEBUG_F32_OUT: fp8bs_gemm_fprop, _dgrad and _wgrad write the FP32
 *     promotion accumulator itself -- float [rows][cols], 4 bytes per
 *     element in the same output pointer -- instead of its BF16 rounding, so
 *     that a test can compare the tensor-core partial sums and the promotion
 *     chain with a reference without the BF16 step.  Other entry points
 *     ignore it.  FP8BS_ERR_INVALID_ARG for unknown bits.
 *   fp8bs_debug_occupy_sms: launches `ctas` (1 .. SM count) CTAs on `stream`
 *     that each hold one SM -- their shared memory leaves no room for a GEMM
 *     CTA -- for `ns` nanoseconds (at most 2e9), then exit: for testing that
 *     a GEMM on another stream completes while part of the GPU is busy.
 *   fp8bs_debug_split_plan: the split-K plan for `tiles` output tiles of
 *     `kblocks` 128-wide contraction blocks on `sms` SMs, host only (no
 *     device needed): out[0] splits (1 = none), out[1] the first split tile
 *     (tiles before it are whole), out[2] work units, out[3] scratch bytes.
 *     FP8BS_ERR_INVALID_ARG for non-positive sizes or a NULL `out`.
 *   fp8bs_debug_tile_order: the tile order a GEMM launch would use, host
 *     only: the output's m_tiles x n_tiles tiles (128 x 256), contraction of
 *     kc bytes per operand row, split plan (`splits`, `tail_first` as
 *     fp8bs_debug_split_plan gives them), `grid` persistent CTAs, an L2 of
 *     `l2_bytes` and `out_bytes` (1, 2 or 4) per output element.  The GEMMs
 *     take tiles in column strips out[0] tiles wide (row-major inside a
 *     strip; out[0] == n_tiles is plain row-major), the width with the
 *     fewest DRAM bytes of operand panels by a wave-by-wave L2 reuse
 *     estimate: out[1] those bytes for the chosen order, out[2] for
 *     row-major.  FP8BS_ERR_INVALID_ARG for non-positive sizes, more than
 *     2^30 tiles, a bad split or `out_bytes`, or a NULL `out`.
 */
int fp8bs_debug_set_wait_timeout_ns(int64_t ns);
#define FP8BS_DEBUG_F32_OUT 1u
int fp8bs_debug_set_flags(unsigned flags);
int fp8bs_debug_occupy_sms(int ctas, int64_t ns, void* stream);
int fp8bs_debug_force_tile_order(int strip);
int fp8bs_debug_set_fault(int mode);
int fp8bs_debug_e4m3_encode_bits(uint32_t first, int64_t n, uint8_t* out, void* stream);
int fp8bs_debug_split_plan(int64_t tiles, int64_t kblocks, int sms, int64_t* out);
int fp8bs_debug_tile_order(int64_t m_tiles, int64_t n_tiles, int64_t kc, int32_t splits, int64_t tail_first,
                           int64_t grid, int64_t l2_bytes, int32_t out_bytes, int64_t* out);
int fp8bs_debug_silu_mul(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* h, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H_ */
