// quant.cuh -- HBM-bound fused amax + scale + E4M3 cast for the three tile
// shapes of the fine-grained block quantization (1x128 activation tiles,
// 128x1 token-dim tiles written transposed, 128x128 weight blocks).
//
// One CTA owns one 128x128 BF16 tile of the input (32 KB): it copies the
// tile into shared memory with 16-byte cp.async copies (no staging
// registers, so five CTAs fit on an SM and their load, compute and store
// phases overlap), then computes
//   - row maxima (1x128 tiles) with a bank-skewed row sweep,
//   - column maxima (128x1 tiles, or the 128x128 block) with a column sweep,
// on the BF16 bit patterns (|x| ordering equals the ordering of the
// sign-cleared bits, so a packed 16-bit unsigned max is exact), then one
// IEEE division pair per tile for s = amax/448 and inv = 448/amax, then
// the cast q = E4M3_rne_satfinite(x * inv) and packed, coalesced stores.
// Because every stored value is an exact function of the BF16 input (an
// exact max, correctly rounded divisions and multiply, a correctly rounded
// conversion), the output is bit-identical to a scalar implementation of
// the same formulas.
#pragma once

#include <cfloat>
#include <cstdint>

#include "ptx.cuh"

namespace fp8bs {

enum : int { QM_ROW = 1, QM_COLT = 2, QM_BLOCK = 4 };

// Four E4M3 codes from the low (lo = true) or high BF16 halves of four words.
__device__ __forceinline__ uint32_t e4m3x4_half(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, float iv,
                                                bool lo) {
    const float a = lo ? bf16lo_to_f32(w0) : bf16hi_to_f32(w0);
    const float b = lo ? bf16lo_to_f32(w1) : bf16hi_to_f32(w1);
    const float c = lo ? bf16lo_to_f32(w2) : bf16hi_to_f32(w2);
    const float d = lo ? bf16lo_to_f32(w3) : bf16hi_to_f32(w3);
    return e4m3x2(__fmul_rn(a, iv), __fmul_rn(b, iv)) | (e4m3x2(__fmul_rn(c, iv), __fmul_rn(d, iv)) << 16);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// x: BF16 [rows][cols] viewed as 32-bit words (two BF16 per word); ld is
// the token leading dimension of the token-major outputs, rows rounded up
// to 128 (the grid covers ld/128 row blocks; rows past `rows` read as zeros).
// MODE & QM_ROW   : q [rows][cols], s [cols/128][ld]
// MODE & QM_COLT  : qT [cols][ld], sT [ld/128][cols]
// MODE == QM_BLOCK: q [rows][cols], qT [cols][rows] (nullable),
//                   s [rows/128][cols/128]   (rows % 128 == 0, ld == rows)
template <int MODE>
__global__ void __launch_bounds__(256, 5) quant_tile_kernel(const uint32_t* __restrict__ x, int64_t rows,
                                                            int64_t cols, int64_t ld, uint8_t* __restrict__ q,
                                                            float* __restrict__ s, uint8_t* __restrict__ qT,
                                                            float* __restrict__ sT) {
    constexpr bool kRow = (MODE & QM_ROW) != 0;
    constexpr bool kColT = (MODE & QM_COLT) != 0;
    constexpr bool kBlock = (MODE & QM_BLOCK) != 0;
    constexpr bool kNeedCol = kColT || kBlock;

    __shared__ __align__(16) uint32_t tile[128 * 64];
    __shared__ uint32_t rmax[128];
    __shared__ float rinv[128];
    __shared__ uint32_t cpart[4][64];
    __shared__ float cinv[128];
    __shared__ float binv;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;
    const int64_t wpr = cols >> 1;  // words per row

    // 1. The 128x128 tile into shared memory: 2048 chunks of 16 bytes, eight
    //    per thread, all in flight at once; rows past the end are zeros.
    const bool full = r0 + 128 <= rows;  // every tile but a token tail's last
    {
        const uint32_t* src = x + r0 * wpr + (c0 >> 1);
        const uint32_t dst = smem_u32(tile);
        if (full) {
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int id = i * 256 + tid, r = id >> 4, ch = id & 15;
                cp_async16(dst + static_cast<uint32_t>(r * 256 + ch * 16), src + r * wpr + ch * 4);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int id = i * 256 + tid, r = id >> 4, ch = id & 15;
                if (r0 + r < rows)
                    cp_async16(dst + static_cast<uint32_t>(r * 256 + ch * 16), src + r * wpr + ch * 4);
                else
                    *reinterpret_cast<uint4*>(&tile[r * 64 + ch * 4]) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
    __syncthreads();

    // 2a. Column sweep: thread -> column pair cp (columns 2cp, 2cp+1), rows
    //     [32 seg, 32 seg + 32).  Lanes read consecutive words: no conflicts.
    const int cp = tid & 63, seg = tid >> 6;
    if constexpr (kNeedCol) {
        uint32_t m = 0;
#pragma unroll 8
        for (int i = 0; i < 32; i++) m = max_u16x2(m, tile[(seg * 32 + i) * 64 + cp] & 0x7FFF7FFFu);
        cpart[seg][cp] = m;
    }
    // 2b. Row sweep: thread -> row tid/2, half tid%2; word order skewed by
    //     lane so the 32 lanes hit 32 different banks.
    if constexpr (kRow) {
        const int r = tid >> 1, h = tid & 1;
        uint32_t m = 0;
#pragma unroll 8
        for (int j = 0; j < 32; j++) m = max_u16x2(m, tile[r * 64 + h * 32 + ((j + lane) & 31)] & 0x7FFF7FFFu);
        m = max_u16x2(m, __shfl_xor_sync(0xffffffffu, m, 1));
        if (h == 0) rmax[r] = max(m & 0xFFFFu, m >> 16);
    }
    __syncthreads();

    // 3. Scales: one division pair per tile, spread over 128 threads.
    if constexpr (kRow) {
        if (tid < 128) {
            float sc, iv;
            tile_scale(__uint_as_float(rmax[tid] << 16), sc, iv);
            rinv[tid] = iv;
            s[static_cast<int64_t>(blockIdx.x) * ld + r0 + tid] = sc;
        }
    }
    if constexpr (kColT) {
        if (tid < 128) {
            const int p = tid >> 1;
            uint32_t m = max_u16x2(max_u16x2(cpart[0][p], cpart[1][p]), max_u16x2(cpart[2][p], cpart[3][p]));
            const uint32_t bits = (tid & 1) ? (m >> 16) : (m & 0xFFFFu);
            float sc, iv;
            tile_scale(__uint_as_float(bits << 16), sc, iv);
            cinv[tid] = iv;
            sT[static_cast<int64_t>(blockIdx.y) * cols + c0 + tid] = sc;
        }
    }
    if constexpr (kBlock) {
        if (warp == 0) {
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) m = max_u16x2(m, (&cpart[0][0])[i * 32 + lane]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = max_u16x2(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) {
                float sc, iv;
                tile_scale(__uint_as_float(max(m & 0xFFFFu, m >> 16) << 16), sc, iv);
                binv = iv;
                s[static_cast<int64_t>(blockIdx.y) * (cols >> 7) + blockIdx.x] = sc;
            }
        }
    }
    __syncthreads();

    // 4a. Row-layout payload (1x128 tiles, or the weight block): warp w
    //     writes rows [16w, 16w+16), lane l owns elements [4l, 4l+4): one
    //     128-byte store per row.
    if constexpr (kRow || kBlock) {
        auto row_out = [&](int r) {
            const uint2 w2 = *reinterpret_cast<const uint2*>(&tile[r * 64 + 2 * lane]);
            const float iv = kRow ? rinv[r] : binv;
            const uint32_t lo = e4m3x2(__fmul_rn(bf16lo_to_f32(w2.x), iv), __fmul_rn(bf16hi_to_f32(w2.x), iv));
            const uint32_t hi = e4m3x2(__fmul_rn(bf16lo_to_f32(w2.y), iv), __fmul_rn(bf16hi_to_f32(w2.y), iv));
            *reinterpret_cast<uint32_t*>(q + (r0 + r) * cols + c0 + 4 * lane) = lo | (hi << 16);
        };
        if (full) {
#pragma unroll 4
            for (int i = 0; i < 16; i++) row_out(warp * 16 + i);
        } else {
            for (int i = 0; i < 16 && r0 + warp * 16 + i < rows; i++) row_out(warp * 16 + i);
        }
    }

    // 4b. Transposed payload: thread (cp, seg) converts 32 tokens of columns
    //     2cp and 2cp+1 (re-reading the column words from shared memory),
    //     then, once every read of the tile is done, parks its 2 x 32 bytes
    //     in the tile buffer as rows of a [128 columns][128 tokens] byte
    //     block (row stride 144 bytes, which spreads both the parking writes
    //     and the reads below over all banks), and the CTA writes that block
    //     out as full 128-byte lines of qT.
    if constexpr (kNeedCol) {
        if (kColT || qT != nullptr) {
            const float ivl = kColT ? cinv[2 * cp] : binv;
            const float ivh = kColT ? cinv[2 * cp + 1] : binv;
            uint4 pl[2], ph[2];
#pragma unroll
            for (int g = 0; g < 2; g++) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; i++) w[i] = tile[(seg * 32 + g * 16 + i) * 64 + cp];
                pl[g].x = e4m3x4_half(w[0], w[1], w[2], w[3], ivl, true);
                pl[g].y = e4m3x4_half(w[4], w[5], w[6], w[7], ivl, true);
                pl[g].z = e4m3x4_half(w[8], w[9], w[10], w[11], ivl, true);
                pl[g].w = e4m3x4_half(w[12], w[13], w[14], w[15], ivl, true);
                ph[g].x = e4m3x4_half(w[0], w[1], w[2], w[3], ivh, false);
                ph[g].y = e4m3x4_half(w[4], w[5], w[6], w[7], ivh, false);
                ph[g].z = e4m3x4_half(w[8], w[9], w[10], w[11], ivh, false);
                ph[g].w = e4m3x4_half(w[12], w[13], w[14], w[15], ivh, false);
            }
            constexpr int kStride = 144;  // bytes per parked qT row
            uint8_t* park = reinterpret_cast<uint8_t*>(tile);
            __syncthreads();  // every read of the BF16 tile is done
#pragma unroll
            for (int g = 0; g < 2; g++) {
                *reinterpret_cast<uint4*>(park + (2 * cp) * kStride + seg * 32 + g * 16) = pl[g];
                *reinterpret_cast<uint4*>(park + (2 * cp + 1) * kStride + seg * 32 + g * 16) = ph[g];
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int id = i * 256 + tid, rr = id >> 3, part = id & 7;
                const uint4 v = *reinterpret_cast<const uint4*>(park + rr * kStride + part * 16);
                *reinterpret_cast<uint4*>(qT + (c0 + rr) * ld + r0 + part * 16) = v;
            }
        }
    }
}

// FP32 bit patterns [first, first+n) -> E4M3 codes, through the same
// conversion the quantizers use (pairs of values per instruction).
__global__ void e4m3_encode_bits_kernel(uint32_t first, int64_t n, uint8_t* __restrict__ out) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 4;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4; i < n; i += stride) {
        const uint32_t b = first + static_cast<uint32_t>(i);
        if (i + 4 <= n) {
            const uint32_t lo = e4m3x2(__uint_as_float(b), __uint_as_float(b + 1));
            const uint32_t hi = e4m3x2(__uint_as_float(b + 2), __uint_as_float(b + 3));
            *reinterpret_cast<uint32_t*>(out + i) = lo | (hi << 16);
        } else {
            for (int64_t j = i; j < n; j++)
                out[j] = static_cast<uint8_t>(e4m3x2(__uint_as_float(first + static_cast<uint32_t>(j)), 0.0f));
        }
    }
}

}  // namespace fp8bs
