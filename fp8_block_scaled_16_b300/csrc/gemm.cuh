// gemm.cuh -- FP8 block-scaled GEMM with per-128-K promotion on tcgen05.
//
// C[i][j] = bf16( fma-chain over 128-blocks b of P_b[i][j] * (sa[b][i] * sb(b, j)) )
// P_b[i][j] = sum_{k in block b} A[i][k] * B[j][k]   (A, B: E4M3, K-major)
//
// The scheme's per-block FP32 scales are arbitrary FP32 values, so the
// tensor core's block-scaled (UE8M0, 32-element) MMA cannot apply them;
// each 128-K block's partial sum therefore lands in its own TMEM buffer and
// is promoted in registers, as the DeepSeek-V3 scheme the Puro-2B pages
// follow prescribes (blog section "FP8：加快 RTX 5090 上的训练"; arXiv part
// 1/7, section 2.1).
//
// Persistent kernel, one 384-thread CTA per SM, 128x256 output tiles:
//   warp 0 (one lane): TMA producer -- A tile 128x128 B and B tile 256x128 B
//       per K block into a STAGES-deep shared-memory ring (128-byte
//       swizzle), plus the K block's row scales (and, for the weight
//       gradient, its 256 column scales) into a separate scale ring;
//   warp 1 (one lane): MMA issuer -- four tcgen05.mma (K = 32 each) per K
//       block into one of two 128x256 FP32 TMEM buffers (512 columns), the
//       first with accumulate off, then commits to free the smem stage and
//       to publish the buffer;
//   warps 2, 3: idle (they complete the first warpgroup, whose registers
//       are handed to the epilogue warpgroups with setmaxnreg);
//   warps 4..11: promotion + epilogue -- each warp owns a 32-lane TMEM
//       quadrant (rows) and one 128-column half; per K block it loads its
//       32x128 partial with tcgen05.ld, releases the buffer, and does
//       acc = fma(P_b, sa*sb, acc) on 128 FP32 registers per thread; at the
//       end of a tile it rounds to BF16 and stores.
// While the epilogue promotes block b, the tensor cores already compute
// block b+1 into the other buffer.
//
// Every mbarrier wait is bounded (see WaitCtx): on expiry the CTA records
// a timeout in the device status word, waits (bounded) for its own copies
// and MMAs in flight, frees its TMEM and returns.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace fp8bs {
namespace gemm {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int STAGES = 4;
constexpr int SSLOTS = 8;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SA_FLOATS = BM;
constexpr int SB_FLOATS = BN;
constexpr int SLOT_FLOATS = SA_FLOATS + SB_FLOATS;
constexpr int NUM_EPI_WARPS = 8;
constexpr int THREADS = 128 + NUM_EPI_WARPS * 32;
// Register split after launch (launch: 168 per thread = 384 x 168 total).
// Per SM sub-partition: one first-warpgroup warp and two epilogue warps,
// 48 + 2 x 224 = 496 <= 512 registers per lane slot; CTA-wide
// 128 x 48 + 256 x 224 = 63488 <= 64512.
constexpr int REGS_CTRL = 48;
constexpr int REGS_EPI = 224;
constexpr uint32_t TMEM_COLS = 2 * BN;

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_SCALE = OFF_B + STAGES * B_BYTES;
constexpr int OFF_BAR = OFF_SCALE + SSLOTS * SLOT_FLOATS * 4;
constexpr int NUM_BARS = 2 * STAGES + 4 + 2 * SSLOTS;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1024-byte alignment

static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(THREADS == 384, "warp roles");
static_assert(128 * REGS_CTRL + NUM_EPI_WARPS * 32 * REGS_EPI <= THREADS * 168, "register split");

enum : int { SB_SCALAR = 0, SB_VECTOR = 1 };

struct Params {
    int32_t m_tiles, n_tiles, kblocks;
    int32_t nb_valid;             // number of 128-column blocks of the output (cols / 128)
    int64_t cols;                 // output row length
    const float* sb;              // SB_SCALAR: scalar B-scale table
    int64_t sb_stride_j;          // ... index = jb * sb_stride_j + b * sb_stride_b
    int64_t sb_stride_b;
    uint16_t* out;                // BF16 [rows][cols]
    uint32_t* status;
    uint64_t timeout_ns;
    int32_t fault;                // test hook: withhold CTA 0's first operand copy
};

__device__ __forceinline__ uint32_t bar_full(int s) { return s; }
__device__ __forceinline__ uint32_t bar_empty(int s) { return STAGES + s; }
__device__ __forceinline__ uint32_t bar_tfull(int b) { return 2 * STAGES + b; }
__device__ __forceinline__ uint32_t bar_tempty(int b) { return 2 * STAGES + 2 + b; }
__device__ __forceinline__ uint32_t bar_sfull(int i) { return 2 * STAGES + 4 + i; }
__device__ __forceinline__ uint32_t bar_sempty(int i) { return 2 * STAGES + 4 + SSLOTS + i; }

// Bounded wait used while tearing down after an abort: ignores the abort
// flag, only the time limit ends it.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > timeout_ns) return;
    }
}

// acc[base + i] = fma(P[i], sc, acc[base + i]) for one 32-column chunk.
__device__ __forceinline__ void promote_scalar(float (&acc)[128], int base, const uint32_t (&r)[32], float sc) {
#pragma unroll
    for (int i = 0; i < 32; i++) acc[base + i] = fmaf(__uint_as_float(r[i]), sc, acc[base + i]);
}

// Rank-1 block scale (weight gradient): the FP32 product sa * sb[j] is
// rounded first, then fused into the accumulator, as for a scalar scale.
__device__ __forceinline__ void promote_vector(float (&acc)[128], int base, const uint32_t (&r)[32], float sa,
                                               const float* sbv) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        const float4 s4 = *reinterpret_cast<const float4*>(sbv + base + i);
        acc[base + i + 0] = fmaf(__uint_as_float(r[i + 0]), __fmul_rn(sa, s4.x), acc[base + i + 0]);
        acc[base + i + 1] = fmaf(__uint_as_float(r[i + 1]), __fmul_rn(sa, s4.y), acc[base + i + 1]);
        acc[base + i + 2] = fmaf(__uint_as_float(r[i + 2]), __fmul_rn(sa, s4.z), acc[base + i + 2]);
        acc[base + i + 3] = fmaf(__uint_as_float(r[i + 3]), __fmul_rn(sa, s4.w), acc[base + i + 3]);
    }
}

template <int SBMODE>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + OFF_BAR;
    auto bar = [&](uint32_t i) { return bar0 + 8u * i; };
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + OFF_MISC);  // [0] TMEM base, [1] abort flag

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(bar(bar_full(s)), 1);
            mbar_init(bar(bar_empty(s)), 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(bar(bar_tfull(b)), 1);
            mbar_init(bar(bar_tempty(b)), NUM_EPI_WARPS);
        }
        for (int i = 0; i < SSLOTS; i++) {
            mbar_init(bar(bar_sfull(i)), 1);
            mbar_init(bar(bar_sempty(i)), NUM_EPI_WARPS);
        }
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSA);
        if (SBMODE == SB_VECTOR) tma_prefetch_desc(&tmSB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&misc[0]), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem = misc[0];
    const WaitCtx wc{reinterpret_cast<volatile uint32_t*>(&misc[1]), p.status, p.timeout_ns};
    const int num_tiles = p.m_tiles * p.n_tiles;
    const int kblocks = p.kblocks;

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CTRL));
      if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0, slot = 0;
            uint32_t ph = 0, sph = 0;
            uint32_t armed = 0, armed_par = 0, inj = 0;      // per stage
            uint32_t sarmed = 0, sarmed_par = 0;             // per scale slot
            bool ok = true;
            constexpr uint32_t kScaleBytes = (SA_FLOATS + (SBMODE == SB_VECTOR ? SB_FLOATS : 0)) * 4;
            for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
                const int mb = t / p.n_tiles, nb = t - mb * p.n_tiles;
                for (int kb = 0; kb < kblocks; kb++) {
                    if (!wait_bounded(bar(bar_empty(stage)), ph ^ 1u, wc)) { ok = false; break; }
                    const uint32_t fb = bar(bar_full(stage));
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    const bool inject = p.fault != 0 && blockIdx.x == 0 && t == static_cast<int>(blockIdx.x) && kb == 0;
                    if (!inject) {
                        tma_load_2d(sbase + OFF_A + stage * A_BYTES, &tmA, kb * BK, mb * BM, fb);
                        tma_load_2d(sbase + OFF_B + stage * B_BYTES, &tmB, kb * BK, nb * BN, fb);
                        inj &= ~(1u << stage);
                    } else {
                        inj |= 1u << stage;
                    }
                    armed |= 1u << stage;
                    armed_par = (armed_par & ~(1u << stage)) | (ph << stage);
                    if (++stage == STAGES) { stage = 0; ph ^= 1u; }

                    if (!wait_bounded(bar(bar_sempty(slot)), sph ^ 1u, wc)) { ok = false; break; }
                    const uint32_t sfb = bar(bar_sfull(slot));
                    const uint32_t sdst = sbase + OFF_SCALE + slot * SLOT_FLOATS * 4;
                    mbar_arrive_expect_tx(sfb, kScaleBytes);
                    tma_load_2d(sdst, &tmSA, mb * BM, kb, sfb);
                    if (SBMODE == SB_VECTOR) tma_load_2d(sdst + SA_FLOATS * 4, &tmSB, nb * BN, kb, sfb);
                    sarmed |= 1u << slot;
                    sarmed_par = (sarmed_par & ~(1u << slot)) | (sph << slot);
                    if (++slot == SSLOTS) { slot = 0; sph ^= 1u; }
                }
            }
            if (!ok) {
                // Let every copy this CTA issued land before it exits.
                for (int s = 0; s < STAGES; s++)
                    if (((armed >> s) & 1u) && !((inj >> s) & 1u))
                        drain_wait(bar(bar_full(s)), (armed_par >> s) & 1u, p.timeout_ns);
                for (int i = 0; i < SSLOTS; i++)
                    if ((sarmed >> i) & 1u) drain_wait(bar(bar_sfull(i)), (sarmed_par >> i) & 1u, p.timeout_ns);
            }
        }
      } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
            int stage = 0, tb = 0;
            uint32_t ph = 0, tph = 0;
            bool ok = true, issued = false;
            int last_tb = 0;
            uint32_t last_tph = 0;
            for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
                for (int kb = 0; kb < kblocks; kb++) {
                    if (!wait_bounded(bar(bar_tempty(tb)), tph ^ 1u, wc)) { ok = false; break; }
                    tc_fence_after();
                    if (!wait_bounded(bar(bar_full(stage)), ph, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = sbase + OFF_A + stage * A_BYTES;
                    const uint32_t b0 = sbase + OFF_B + stage * B_BYTES;
                    const uint32_t d = tmem + static_cast<uint32_t>(tb * BN);
#pragma unroll
                    for (int kk = 0; kk < BK / 32; kk++)
                        mma_f8(d, sdesc_k_major_sw128(a0 + kk * 32), sdesc_k_major_sw128(b0 + kk * 32), idesc,
                               kk > 0 ? 1u : 0u);
                    mma_commit(bar(bar_empty(stage)));
                    mma_commit(bar(bar_tfull(tb)));
                    issued = true;
                    last_tb = tb;
                    last_tph = tph;
                    if (++stage == STAGES) { stage = 0; ph ^= 1u; }
                    tb ^= 1;
                    if (tb == 0) tph ^= 1u;
                }
            }
            if (!ok && issued) drain_wait(bar(bar_tfull(last_tb)), last_tph, p.timeout_ns);
        }
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_EPI));
        // ------------------------------------------------ promotion + epilogue
        const int ew = warp - 4;
        const int quad = warp & 3;   // TMEM lanes this warp may access
        const int half = ew >> 2;    // 128-column half of the tile
        const int row = quad * 32 + lane;
        const float* ring = reinterpret_cast<const float*>(smem + OFF_SCALE);
        int tb = 0, slot = 0;
        uint32_t tph = 0, sph = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
            const int mb = t / p.n_tiles, nb = t - mb * p.n_tiles;
            const int jb = nb * 2 + half;
            const bool jvalid = jb < p.nb_valid;
            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; i++) acc[i] = 0.0f;
            float sb_next = 0.0f;
            if (SBMODE == SB_SCALAR && jvalid) sb_next = __ldg(p.sb + jb * p.sb_stride_j);
            for (int kb = 0; kb < kblocks; kb++) {
                const float sb_cur = sb_next;
                if (SBMODE == SB_SCALAR && jvalid && kb + 1 < kblocks)
                    sb_next = __ldg(p.sb + jb * p.sb_stride_j + (kb + 1) * p.sb_stride_b);
                if (!warp_wait_bounded(bar(bar_sfull(slot)), sph, wc)) { ok = false; break; }
                const float* sl = ring + slot * SLOT_FLOATS;
                const float sa = sl[row];
                if (!warp_wait_bounded(bar(bar_tfull(tb)), tph, wc)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) +
                                       static_cast<uint32_t>(tb * BN + half * 128);
                // Chunk c+1's TMEM load is in flight while chunk c is promoted.
                uint32_t ra[32], rb[32];
                if (SBMODE == SB_SCALAR) {
                    const float sc = __fmul_rn(sa, sb_cur);
                    tmem_ld_32cols(taddr + 0, ra);
                    tmem_wait_ld(ra);
                    tmem_ld_32cols(taddr + 32, rb);
                    promote_scalar(acc, 0, ra, sc);
                    tmem_wait_ld(rb);
                    tmem_ld_32cols(taddr + 64, ra);
                    promote_scalar(acc, 32, rb, sc);
                    tmem_wait_ld(ra);
                    tmem_ld_32cols(taddr + 96, rb);
                    promote_scalar(acc, 64, ra, sc);
                    tmem_wait_ld(rb);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(bar_tempty(tb)));
                    promote_scalar(acc, 96, rb, sc);
                } else {
                    const float* sbv = sl + SA_FLOATS + half * 128;
                    tmem_ld_32cols(taddr + 0, ra);
                    tmem_wait_ld(ra);
                    tmem_ld_32cols(taddr + 32, rb);
                    promote_vector(acc, 0, ra, sa, sbv);
                    tmem_wait_ld(rb);
                    tmem_ld_32cols(taddr + 64, ra);
                    promote_vector(acc, 32, rb, sa, sbv);
                    tmem_wait_ld(ra);
                    tmem_ld_32cols(taddr + 96, rb);
                    promote_vector(acc, 64, ra, sa, sbv);
                    tmem_wait_ld(rb);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(bar_tempty(tb)));
                    promote_vector(acc, 96, rb, sa, sbv);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(bar_sempty(slot)));
                tb ^= 1;
                if (tb == 0) tph ^= 1u;
                if (++slot == SSLOTS) { slot = 0; sph ^= 1u; }
            }
            if (!ok) break;
            if (jvalid) {
                uint16_t* orow = p.out + (static_cast<int64_t>(mb) * BM + row) * p.cols + static_cast<int64_t>(jb) * 128;
#pragma unroll
                for (int j = 0; j < 128; j += 8) {
                    uint4 v;
                    v.x = f32x2_to_bf16x2(acc[j + 0], acc[j + 1]);
                    v.y = f32x2_to_bf16x2(acc[j + 2], acc[j + 3]);
                    v.z = f32x2_to_bf16x2(acc[j + 4], acc[j + 5]);
                    v.w = f32x2_to_bf16x2(acc[j + 6], acc[j + 7]);
                    *reinterpret_cast<uint4*>(orow + j) = v;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace gemm
}  // namespace fp8bs
