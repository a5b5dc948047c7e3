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
// Persistent kernel, one 384-thread CTA per SM, 128 x 256 output tiles, K
// block 128; the warps' loops run converged and one lane issues the TMA and
// tcgen05 instructions:
//   warp 0: TMA producer -- A tile 128x128 B and B tile 256x128 B per K block
//       into a 3-stage shared-memory ring (128-byte swizzle);
//   warp 1: MMA issuer -- four tcgen05.mma (K = 32 each) per K block into one
//       of two 128 x 256 FP32 TMEM buffers (all 512 columns), the first with
//       accumulate off, then one commit whose barrier both frees the smem
//       stage and tells the promotion warps that the buffer is complete;
//   warp 2: scale loader -- into an 8-slot shared-memory ring with cp.async:
//       forward / data gradient, per slot the 128 row scales and the two
//       weight scales of 4 consecutive K blocks; weight gradient, per slot
//       one K block's 128 row scales and 256 column scales (regrouped for
//       the epilogue's layout);
//   warp 3: output store issuer -- for whole tiles with a plain BF16
//       output, the tile's TMA stores once every promotion warp has staged
//       its slice, so that the promotion warps start the next tile at once;
//   warps 4..11: promotion + epilogue -- each warp owns a 32-lane TMEM
//       quadrant (rows) and one 128-column half; per K block it loads its
//       partial with tcgen05.ld, 64 columns at a time (.32x32b: a row per
//       thread; the weight gradient uses .16x256b: 4 rows x 32 columns per
//       thread, fewer column scales to load), releases the TMEM buffer after
//       the last load, and does acc = fma(P_b, sa*sb, acc) with packed FP32
//       FMAs on 128 registers per thread; at the end of a tile it writes the
//       result through swizzled shared staging and TMA: BF16 stores, FP32
//       reduce-adds for an accumulating weight gradient, and/or, for a
//       forward product, the output's 1x128 E4M3 quantization (a thread's
//       128 columns are one whole tile); for a gate+up product, H =
//       SiLU(G) * U and its 1x128 quantization, the gate and the up warp of
//       a row each computing half of H.
// While the epilogue promotes block b, the tensor cores already compute
// block b+1 into the other buffer.
//
// Work comes in units (tile, K range): one per tile, or, where the last wave
// of tiles would leave many SMs idle, 2-8 splits of the contraction of some
// or all tiles, whose FP32 partials meet in caller-provided scratch (see
// Params::splits).  One launch may compute several products (Group): their
// units are dealt to the persistent CTAs as one list.  Tiles are taken in
// column strips Params::strip tiles wide (row-major when strip == n_tiles),
// a width the host picks per shape to limit DRAM re-reads of operand
// panels; only which tiles a split plan splits depends on it.  Rows past the
// output's last row (a token count that is not a multiple of 128) read zeros
// through TMA and are not stored.
//
// The scale ring is written with cp.async (generic proxy) rather than TMA:
// the epilogue reads it with ordinary loads, and a TMA write into a slot
// those loads have just released would need a proxy fence per K block.
//
// Every wait is bounded (see WaitCtx): on expiry the CTA records a timeout
// in the device status word, waits (bounded) for its own copies and MMAs in
// flight, frees its TMEM and returns.
#pragma once

#include <cstdint>

#include "act.cuh"
#include "ptx.cuh"

namespace fp8bs {
namespace gemm {

constexpr int BM = 128, BK = 128;
constexpr int SSLOTS = 8;
constexpr int NUM_EPI_WARPS = 8;
constexpr int THREADS = 128 + NUM_EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
static_assert(THREADS == 384, "warp roles");

enum : int { SB_SCALAR = 0, SB_VECTOR = 1 };

// Register split after launch (168 per thread at launch, 384 x 168 = 64512 in
// all): `ctrl` for the four first-warpgroup warps, `epi` for the eight
// promotion warps.  The weight gradient's promotion holds 128 accumulators,
// 64 loaded values and its scales at once; at 224 registers it spills, so its
// kernels give it 232 and the first warpgroup 40.
template <int SBMODE>
struct RegSplit {
    static constexpr int ctrl = SBMODE == SB_VECTOR ? 40 : 48;
    static constexpr int epi = SBMODE == SB_VECTOR ? 232 : 224;
    static_assert(128 * ctrl + NUM_EPI_WARPS * 32 * epi <= THREADS * 168, "register split");
};
// Epilogue variants of the forward product, each its own kernel so that the
// plain kernel carries none of the others' code: the tile as BF16 (or FP32
// reduce-adds); plus its 1x128 FP8 quantization; the SwiGLU block instead.
enum : int { EPI_PLAIN = 0, EPI_FP8 = 1, EPI_SWIGLU = 2 };

// Shared-memory plan for a 128 x BN tile.
template <int BN>
struct Tile {
    static_assert(BN == 256, "tile width");
    static constexpr int NBUF = static_cast<int>(TMEM_COLS) / BN;  // TMEM accumulator buffers
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = 3;
    static constexpr int SA_FLOATS = BM;
    // Weight-gradient column scales, regrouped for the promotion threads: per
    // 128-column half, four groups (one per t%4 of a .16x256b load) of the 32
    // columns such a thread holds, each group padded to 36 floats so that the
    // four groups start in different banks.
    static constexpr int SB_GROUP = 36;
    static constexpr int SB_HALF = 4 * SB_GROUP;
    static constexpr int SB_FLOATS = 2 * SB_HALF;
    // Forward / data gradient: one slot carries the scales of SBATCH K
    // blocks -- row scales [SBATCH][128], then the weight scales of the
    // tile's two 128-column halves [SBATCH][2] -- so the promotion warps
    // synchronise on the ring once per SBATCH blocks.
    static constexpr int SBATCH = 4;
    static constexpr int SCALAR_SLOT_FLOATS = SBATCH * (SA_FLOATS + 2);
    static constexpr int SLOT_FLOATS =
        (SA_FLOATS + SB_FLOATS) > SCALAR_SLOT_FLOATS ? (SA_FLOATS + SB_FLOATS) : SCALAR_SLOT_FLOATS;
    static constexpr int COLS = BN / 2;                           // columns per epilogue warp
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SCALE = OFF_B + STAGES * B_BYTES;
    // Output staging for the TMA store: per epilogue warp two 32-row x
    // 64-column BF16 boxes (4 KB each, 128-byte swizzle).
    static constexpr int OUT_BOX_BYTES = 32 * 64 * 2;
    static constexpr int OFF_OUT = (OFF_SCALE + SSLOTS * SLOT_FLOATS * 4 + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_OUT + NUM_EPI_WARPS * 2 * OUT_BOX_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + NBUF + 2 * SSLOTS + 14;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    // SwiGLU epilogue: per quadrant and column half, the 32 rows' partial amax
    // of H as BF16 bits (H is BF16, so its amax is too).
    static constexpr int OFF_AMAX = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = OFF_AMAX + 4 * 2 * 32 * 2 + 1024;  // + slack for 1024-byte alignment
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "stage alignment for 128-byte swizzle");
    static_assert(COLS == 128, "epilogue chunking assumes 128 columns per warp");
    static_assert(SB_FLOATS >= BN && (SA_FLOATS + SB_FLOATS) % 4 == 0 && SLOT_FLOATS % 4 == 0, "scale slot layout");
    static_assert(OFF_OUT % 1024 == 0, "swizzled staging alignment");
    // barrier indices
    static __device__ __forceinline__ uint32_t full(int s) { return s; }
    static __device__ __forceinline__ uint32_t empty(int s) { return STAGES + s; }
    // empty(s) completes when the MMAs that read stage s have finished: it
    // frees the stage for the producer and also tells the promotion warps
    // that the accumulator buffer those MMAs wrote is complete.
    static __device__ __forceinline__ uint32_t tempty(int b) { return 2 * STAGES + b; }
    static __device__ __forceinline__ uint32_t sfull(int i) { return 2 * STAGES + NBUF + i; }
    static __device__ __forceinline__ uint32_t sempty(int i) { return 2 * STAGES + NBUF + SSLOTS + i; }
    // SwiGLU epilogue, per quadrant q (the gate and the up warp of its rows):
    // xhalf -- both have staged the half the other needs; xamax -- both have
    // published their partial amax; xq8 -- the up warp's FP8 half is staged.
    static __device__ __forceinline__ uint32_t xhalf(int q) { return 2 * STAGES + NBUF + 2 * SSLOTS + q; }
    static __device__ __forceinline__ uint32_t xamax(int q) { return 2 * STAGES + NBUF + 2 * SSLOTS + 4 + q; }
    static __device__ __forceinline__ uint32_t xq8(int q) { return 2 * STAGES + NBUF + 2 * SSLOTS + 8 + q; }
    // Plain BF16 epilogue with its TMA stores issued by warp 3: ofull -- every
    // promotion warp has staged its slice of the tile; ofree -- those stores
    // have read the staging buffer.
    static __device__ __forceinline__ uint32_t ofull() { return 2 * STAGES + NBUF + 2 * SSLOTS + 12; }
    static __device__ __forceinline__ uint32_t ofree() { return 2 * STAGES + NBUF + 2 * SSLOTS + 13; }
};

struct Params {
    int32_t m_tiles, n_tiles, kblocks;
    // Tile order: column strips `strip` tiles wide, row-major inside a strip
    // (strip == n_tiles: plain row-major), chosen by the host for the fewest
    // estimated DRAM re-reads of A and B panels across waves of tiles.
    int32_t strip;
    int32_t nb_valid;             // number of 128-column blocks of the output (cols / 128)
    int64_t rows, cols;           // output shape (rows need not be a multiple of 128)
    int64_t sa_ld;                // row-scale leading dimension: rows rounded up to 128
    const float* sa;              // row scales, [kblocks][sa_ld]
    const float* sb;              // SB_SCALAR: scalar table, index jb * sb_stride_j + b * sb_stride_b
    int64_t sb_stride_j;          //   (jb = 128-column block of the output, b = K block)
    int64_t sb_stride_b;          // SB_VECTOR: column scales [kblocks][cols]
    uint16_t* out;                // BF16 [rows][cols]
    uint32_t* status;
    uint64_t timeout_ns;
    int32_t fault;                // test hook: withhold CTA 0's first operand copy
    int32_t out_f32_add;          // 0: BF16 store into out; 1: FP32 out += result; 2: FP32 out = result
                                  // (test mode: the unrounded accumulator); tmC is FP32 for 1 and 2
    int32_t out_bf16;             // store the BF16 output (tmC); 0 only with out_q
    // Forward product only: the BF16-rounded output also quantized in 1x128
    // row tiles -- E4M3 payload [rows][cols] through tmQ, FP32 scales
    // out_s[cols/128][sa_ld] (null: not requested).
    float* out_s;
    int32_t out_q;
    // Forward product of a gate+up projection whose weight rows alternate
    // in 128-row blocks (gate block j, then up block j): every output tile's
    // column halves are the gate and up values of one 128-wide block of
    // H = SiLU(gate) * up, which the epilogue computes and stores instead of
    // the tile: BF16 H through tmC (if out_bf16) and its 1x128 quantization
    // through tmQ / out_s, both [rows][cols/2].
    int32_t out_swiglu;
    // K splits (1 = none) of the tiles t >= tail_first (0: of every tile).
    // With T = tiles - tail_first split tiles, each part s of tile t leaves
    // its FP32 partial in ws slot (t - tail_first) * splits + s and then
    // counts itself in arrivals[(t - tail_first) * 8 + warp]; the part that
    // arrives last adds all the partials in part order and stores the
    // tile's slice.  No part waits for another, so the parts need not be
    // resident at the same time.  A counter holds (epoch << 8) | arrivals;
    // a value with another epoch counts as zero, so counters left by
    // earlier launches need no clearing.
    int32_t splits;
    int32_t tail_first;
    float* ws;                    // [T * splits][8 warps][32 float4][32 lanes]
    unsigned long long* arrivals; // [T][8]
    unsigned long long epoch;     // unique per launch, never 0
};

// One unit of work: K blocks [kb0, kb1) of output tile t, part s (split:
// the tile is computed in parts).  Units are numbered whole tiles first
// (t < tail_first), then part 0 of every split tile, then part 1, ...
struct Unit {
    int t, s, kb0, kb1;
    bool split;
};
__device__ __forceinline__ int num_units_of(const Params& p, int num_tiles) {
    return p.tail_first + p.splits * (num_tiles - p.tail_first);
}
// Every role decodes its next unit at each tile boundary, on the path the
// tensor pipe waits on, so whole tiles take no division at all, and split
// parts only 32-bit ones (s < 8 and kblocks < 2^24: s * kblocks < 2^27).
__device__ __forceinline__ Unit unit_of(int u, const Params& p, int num_tiles) {
    Unit w;
    w.s = 0;
    w.split = false;
    w.kb0 = 0;
    w.kb1 = p.kblocks;
    if (p.splits == 1 || u < p.tail_first) {
        w.t = u;
        return w;
    }
    const int v = u - p.tail_first, nt = num_tiles - p.tail_first;
    w.s = v / nt;
    w.t = p.tail_first + v - w.s * nt;
    w.split = true;
    w.kb0 = (w.s * p.kblocks) / p.splits;
    w.kb1 = ((w.s + 1) * p.kblocks) / p.splits;
    return w;
}

// Output tile t's row and column block under the strip order of Params::strip.
__device__ __forceinline__ void tile_coords(int t, const Params& p, int& mb, int& nb) {
    if (p.strip == p.n_tiles) {  // row-major: one division
        mb = t / p.n_tiles;
        nb = t - mb * p.n_tiles;
        return;
    }
    const int per_strip = p.m_tiles * p.strip;
    const int strip = t / per_strip, local = t - strip * per_strip;
    const int width = min(p.strip, p.n_tiles - strip * p.strip);
    mb = local / width;
    nb = strip * p.strip + (local - mb * width);
}

// Up to G products computed by one persistent launch: member g owns the
// work units [first_unit[g], first_unit[g+1]) (its own units numbered as in
// unit_of).  A single product is a group of one.  Every member of a group
// has the same scale mode (the kernel's SBMODE).
constexpr int kGroupMax = 4;
template <int G>
struct Group {
    CUtensorMap tmA[G], tmB[G], tmC[G], tmQ[G];
    Params p[G];
    int32_t count;
    int32_t first_unit[G + 1];
};
template <int G>
__device__ __forceinline__ int member_of(const Group<G>& grp, int u) {
    int g = 0;
    if constexpr (G > 1) {
#pragma unroll
        for (int i = 1; i < G; i++)
            if (i < grp.count && u >= grp.first_unit[i]) g = i;
    }
    return g;
}

// Counts one part of a split tile as arrived and returns the arrivals so
// far, this one included (0 on a failed update, with the CTA's abort flag
// and the device status set).  The counter holds (epoch << 8) | arrivals; a
// value with another epoch is a leftover of an earlier launch and counts as
// zero.  Lock-free: a failed compare-and-swap means another part's update
// succeeded, so with at most 8 parts the loop ends within 8 retries (the cap
// only guards against a corrupted counter).
__device__ __forceinline__ uint32_t count_arrival(unsigned long long* ctr, unsigned long long epoch,
                                                  const WaitCtx& w) {
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(ctr);
    for (int tries = 0; tries < 64; tries++) {
        const unsigned long long next = (cur >> 8) == epoch ? cur + 1 : (epoch << 8) | 1ull;
        const unsigned long long got = atomicCAS(ctr, cur, next);
        if (got == cur) return static_cast<uint32_t>(next & 0xFFull);
        cur = got;
    }
    *w.abort_flag = 1u;
    atomicOr(w.status, kStatusTimeout);
    __threadfence();
    return 0u;
}

// Bounded wait for the warps on the hand-off path, without a warp vote:
// the warp runs converged, and every lane executes the same try_wait on the
// same barrier word (and on the slow path reads the same timer and abort
// flag), so the result is the same in every lane.  The vote of
// warp_wait_bounded costs measurable time on a path the tensor pipe waits on.
__device__ __forceinline__ bool uniform_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bounded(bar, parity, w);
}

// Bounded wait used while tearing down after an abort: ignores the abort
// flag, only the time limit ends it.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > timeout_ns) return;
    }
}

// Orders the uses of `r` after a preceding tcgen05.wait::ld (asm volatile
// statements keep their order, and the uses depend on this one's outputs).
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                   "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// 16-byte global -> shared copy in the generic proxy, completed through
// cp.async.mbarrier.arrive.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// 4- and 8-byte forms (cached at all levels; the only variant with these sizes).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// acc[base + i] = fma(P[i], sc, acc[base + i]) for one 32-column chunk, two
// columns per packed FP32 FMA (each lane of the pair rounds like fmaf).
template <int N>
__device__ __forceinline__ void promote_scalar(float (&acc)[N], int base, const uint32_t (&r)[32], float sc) {
    const float2 s2 = make_float2(sc, sc);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float2 d = __ffma2_rn(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), s2,
                                    make_float2(acc[base + i], acc[base + i + 1]));
        acc[base + i] = d.x;
        acc[base + i + 1] = d.y;
    }
}

// Weight gradient, .16x256b layout: `lo` holds lanes 0-15 and `hi` lanes 16-31
// of the warp's quadrant for the same 64 columns; thread t's rows are
// t/4, t/4+8 (lo) and t/4+16, t/4+24 (hi), with row scales sa4.x..w, and its
// columns 8g + 2(t%4) + {0,1} (g = 0..7), whose scales are cs[2g], cs[2g+1].
// The FP32 product of row and column scale is rounded first, then fused into
// the accumulator, as for a scalar scale.
template <int N>
__device__ __forceinline__ void promote_rank1(float (&acc)[N], int base_lo, int base_hi, const uint32_t (&lo)[32],
                                              const uint32_t (&hi)[32], float4 sa4, const float* cs) {
#pragma unroll
    for (int gp = 0; gp < 4; gp++) {
        const float4 c4 = *reinterpret_cast<const float4*>(cs + 4 * gp);
#pragma unroll
        for (int h2 = 0; h2 < 2; h2++) {
            const int g = 2 * gp + h2;
            const float2 c2 = h2 ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
            const float sr[4] = {sa4.x, sa4.y, sa4.z, sa4.w};
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const uint32_t(&r)[32] = q < 2 ? lo : hi;
                const int i = 4 * g + 2 * (q & 1);
                const int a = (q < 2 ? base_lo : base_hi) + i;
                const float2 sc = __fmul2_rn(make_float2(sr[q], sr[q]), c2);
                const float2 d = __ffma2_rn(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), sc,
                                            make_float2(acc[a], acc[a + 1]));
                acc[a] = d.x;
                acc[a + 1] = d.y;
            }
        }
    }
}

// The plain BF16 epilogue of unit w is staged by the promotion warps and
// stored by warp 3 (the output store issuer) unless the unit is a part of a
// split tile (whose last part, found at run time, stores it) or the output
// is FP32.  Both sides take the same decision from the same unit.
__device__ __forceinline__ bool delegated_store(const Params& p, const Unit& w) {
    return !w.split && p.out_f32_add == 0 && p.out_bf16 != 0;
}

// A promotion warp's 32 x 128 slice of the tile in BF16 into its two
// 32-row x 64-column staging boxes (4 KB each, 128-byte swizzle: the
// 16-byte chunk c of row r at chunk c ^ (r % 8), so the lanes' writes
// spread over all banks), from the .32x32b (SB_SCALAR) or .16x256b
// (SB_VECTOR) accumulator layout.
template <int SBMODE, int N>
__device__ __forceinline__ void stage_bf16_tile(const float (&acc)[N], uint32_t stage_out, int lane) {
    constexpr uint32_t kBox = 32 * 64 * 2;
    if constexpr (SBMODE == SB_SCALAR) {
#pragma unroll
        for (int b = 0; b < 2; b++) {
#pragma unroll
            for (int c = 0; c < 8; c++) {
                const int j = b * 64 + c * 8;
                const uint32_t w0 = f32x2_to_bf16x2(acc[j + 0], acc[j + 1]);
                const uint32_t w1 = f32x2_to_bf16x2(acc[j + 2], acc[j + 3]);
                const uint32_t w2 = f32x2_to_bf16x2(acc[j + 4], acc[j + 5]);
                const uint32_t w3 = f32x2_to_bf16x2(acc[j + 6], acc[j + 7]);
                const uint32_t a = stage_out + static_cast<uint32_t>(b * kBox + lane * 128 + ((c ^ (lane & 7)) << 4));
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                             : "memory");
            }
        }
    } else {
        // .16x256b layout: acc[32L + 4g + 2hi], {+1} is row 16(L/2) + 8hi + t/4,
        // columns 64(L%2) + 8g + 2(t%4) + {0,1}: one BF16 pair per store, the
        // eight rows of a store in eight different 16-byte chunks.
        const int u = lane >> 2, c = lane & 3;
#pragma unroll
        for (int L = 0; L < 4; L++) {
#pragma unroll
            for (int g = 0; g < 8; g++) {
#pragma unroll
                for (int hi = 0; hi < 2; hi++) {
                    const int j = 32 * L + 4 * g + 2 * hi;
                    const int rr = 16 * (L >> 1) + 8 * hi + u;
                    const uint32_t a = stage_out + static_cast<uint32_t>((L & 1) * kBox + rr * 128 + ((g ^ u) << 4) + 4 * c);
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(f32x2_to_bf16x2(acc[j], acc[j + 1])) : "memory");
                }
            }
        }
    }
}

// SwiGLU epilogue helpers (one 64-column half of a warp's 128 accumulator
// columns, offsets fixed at compile time so that acc stays in registers).
// A staging box row is 128 bytes: 16-byte chunk c of row r at c ^ (r % 8).
template <int J0, int N>
__device__ __forceinline__ void stage_bf16_64(const float (&acc)[N], uint32_t box, int lane) {
#pragma unroll
    for (int c = 0; c < 8; c++) {
        const int j = J0 + c * 8;
        const uint32_t a = box + static_cast<uint32_t>(lane * 128 + ((c ^ (lane & 7)) << 4));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(f32x2_to_bf16x2(acc[j], acc[j + 1])),
                     "r"(f32x2_to_bf16x2(acc[j + 2], acc[j + 3])), "r"(f32x2_to_bf16x2(acc[j + 4], acc[j + 5])),
                     "r"(f32x2_to_bf16x2(acc[j + 6], acc[j + 7]))
                     : "memory");
    }
}

// H = bf16(SiLU(G) * U) for acc[J0 .. J0+63] (this warp's gate values if
// GATE, else its up values) with the other operand's BF16 half from `peer`;
// the BF16 H values replace acc and their amax is returned.  Per 8-value
// chunk the four exponentials come first and the eight divisions after, so
// that the exponentials' dependent chains overlap; each value still takes
// the same operations in the same order.
template <int J0, bool GATE, int N>
__device__ __forceinline__ float swiglu_64(float (&acc)[N], uint32_t peer, int lane) {
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < 8; c++) {
        const int j = J0 + c * 8;
        uint32_t pw[4];
        const uint32_t a = peer + static_cast<uint32_t>(lane * 128 + ((c ^ (lane & 7)) << 4));
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(pw[0]), "=r"(pw[1]), "=r"(pw[2]), "=r"(pw[3])
                     : "r"(a)
                     : "memory");
        float2 gv[4], uv[4], dv[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const uint32_t ow = f32x2_to_bf16x2(acc[j + 2 * e], acc[j + 2 * e + 1]);
            const uint32_t gw = GATE ? ow : pw[e];
            const uint32_t uw = GATE ? pw[e] : ow;
            gv[e] = make_float2(bf16lo_to_f32(gw), bf16hi_to_f32(gw));
            uv[e] = make_float2(bf16lo_to_f32(uw), bf16hi_to_f32(uw));
            dv[e] = silu_denom2(gv[e]);
        }
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float2 h = silu_mul2_from_denom(gv[e], dv[e], uv[e]);
            const uint32_t hw = f32x2_to_bf16x2(h.x, h.y);
            acc[j + 2 * e] = bf16lo_to_f32(hw);
            acc[j + 2 * e + 1] = bf16hi_to_f32(hw);
            amax = fmaxf(amax, fmaxf(fabsf(acc[j + 2 * e]), fabsf(acc[j + 2 * e + 1])));
        }
    }
    return amax;
}

// E4M3 codes of acc[J0 .. J0+63] * inv into 16-byte chunks CH0 .. CH0+3 of a
// 128-byte FP8 row.
template <int J0, int CH0, int N>
__device__ __forceinline__ void stage_fp8_64(const float (&acc)[N], float inv, uint32_t box, int lane) {
#pragma unroll
    for (int c = 0; c < 4; c++) {
        uint32_t wv[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int j = J0 + c * 16 + q * 4;
            wv[q] = e4m3x2(__fmul_rn(acc[j], inv), __fmul_rn(acc[j + 1], inv)) |
                    (e4m3x2(__fmul_rn(acc[j + 2], inv), __fmul_rn(acc[j + 3], inv)) << 16);
        }
        const uint32_t a = box + static_cast<uint32_t>(lane * 128 + (((CH0 + c) ^ (lane & 7)) << 4));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(wv[0]), "r"(wv[1]), "r"(wv[2]),
                     "r"(wv[3])
                     : "memory");
    }
}

template <int SBMODE, int BN, int G, int EPI>
__global__ void __launch_bounds__(THREADS, 1) gemm_kernel(const __grid_constant__ Group<G> grp) {
    static_assert(EPI == EPI_PLAIN || (SBMODE == SB_SCALAR && G == 1), "FP8 epilogues: single forward products");
    using T = Tile<BN>;
    constexpr int STAGES = T::STAGES, NBUF = T::NBUF, COLS = T::COLS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + T::OFF_BAR;
    auto bar = [&](uint32_t i) { return bar0 + 8u * i; };
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + T::OFF_MISC);  // [0] TMEM base, [1] abort flag

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(bar(T::full(s)), 1);
            mbar_init(bar(T::empty(s)), 1);
        }
        for (int b = 0; b < NBUF; b++) mbar_init(bar(T::tempty(b)), NUM_EPI_WARPS);
        for (int q = 0; q < 4; q++) {
            mbar_init(bar(T::xhalf(q)), 2);
            mbar_init(bar(T::xamax(q)), 2);
            mbar_init(bar(T::xq8(q)), 1);
        }
        mbar_init(bar(T::ofull()), NUM_EPI_WARPS);
        mbar_init(bar(T::ofree()), 1);
        for (int i = 0; i < SSLOTS; i++) {
            mbar_init(bar(T::sfull(i)), 32);   // one cp.async arrival per lane of the scale warp
            mbar_init(bar(T::sempty(i)), NUM_EPI_WARPS);
        }
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int g = 0; g < grp.count; g++) {
            tma_prefetch_desc(&grp.tmA[g]);
            tma_prefetch_desc(&grp.tmB[g]);
            tma_prefetch_desc(&grp.tmC[g]);
            if (grp.p[g].out_q) tma_prefetch_desc(&grp.tmQ[g]);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&misc[0]), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem = misc[0];
    const Params& p0 = grp.p[0];   // status word, time limit and test hook are the group's
    const WaitCtx wc{reinterpret_cast<volatile uint32_t*>(&misc[1]), p0.status, p0.timeout_ns};
    const int num_units = grp.first_unit[grp.count];
    // Work unit u: its member's parameters, tile count and (tile, K range).
#define FP8BS_UNIT(u)                                          \
    const int g = member_of(grp, u);                           \
    const Params& p = grp.p[g];                                \
    const int num_tiles = p.m_tiles * p.n_tiles;               \
    const Unit w = unit_of((u) - grp.first_unit[g], p, num_tiles)

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(RegSplit<SBMODE>::ctrl));
      // The producer and MMA warps run their loops with all 32 lanes
      // converged (waits are warp-wide); only lane 0 issues the TMA and
      // tcgen05 instructions.  A lone lane looping while its warp-mates
      // park at the final barrier slows the other warps of its SM
      // sub-partition.
      if (warp == 0) {
        // ------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t ph = 0;
        uint32_t armed = 0, armed_par = 0, inj = 0;      // per stage
        bool ok = true;
        for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
            FP8BS_UNIT(u);
            int mb, nb;
            tile_coords(w.t, p, mb, nb);
            for (int kb = w.kb0; kb < w.kb1; kb++) {
                if (!warp_wait_bounded(bar(T::empty(stage)), ph ^ 1u, wc)) { ok = false; break; }
                const bool inject = p0.fault != 0 && blockIdx.x == 0 && u == static_cast<int>(blockIdx.x) && kb == w.kb0;
                if (lane == 0) {
                    const uint32_t fb = bar(T::full(stage));
                    mbar_arrive_expect_tx(fb, T::STAGE_BYTES);
                    if (!inject) {
                        tma_load_2d(sbase + T::OFF_A + stage * T::A_BYTES, &grp.tmA[g], kb * BK, mb * BM, fb);
                        tma_load_2d(sbase + T::OFF_B + stage * T::B_BYTES, &grp.tmB[g], kb * BK, nb * BN, fb);
                    }
                }
                __syncwarp();
                if (!inject) inj &= ~(1u << stage); else inj |= 1u << stage;
                armed |= 1u << stage;
                armed_par = (armed_par & ~(1u << stage)) | (ph << stage);
                if (++stage == STAGES) { stage = 0; ph ^= 1u; }
            }
        }
        if (!ok && lane == 0) {
            // Let every copy this CTA issued land before it exits.
            for (int s = 0; s < STAGES; s++)
                if (((armed >> s) & 1u) && !((inj >> s) & 1u))
                    drain_wait(bar(T::full(s)), (armed_par >> s) & 1u, p0.timeout_ns);
        }
        __syncwarp();
      } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
        int stage = 0, tb = 0;
        uint32_t ph = 0, tph = 0;
        bool ok = true, issued = false;
        int last_stage = 0;
        uint32_t last_ph = 0;
        for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
            FP8BS_UNIT(u);
            (void)num_tiles;
            for (int kb = w.kb0; kb < w.kb1; kb++) {
                // The operands are usually in place long before the buffer is free.
                if (!uniform_wait(bar(T::full(stage)), ph, wc)) { ok = false; break; }
                if (!uniform_wait(bar(T::tempty(tb)), tph ^ 1u, wc)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a0 = sbase + T::OFF_A + stage * T::A_BYTES;
                    const uint32_t b0 = sbase + T::OFF_B + stage * T::B_BYTES;
                    const uint32_t d = tmem + static_cast<uint32_t>(tb * BN);
#pragma unroll
                    for (int kk = 0; kk < BK / 32; kk++)
                        mma_f8(d, sdesc_k_major_sw128(a0 + kk * 32), sdesc_k_major_sw128(b0 + kk * 32), idesc,
                               kk > 0 ? 1u : 0u);
                    // One commit per K block: its barrier frees the stage and
                    // tells the promotion warps that the buffer is complete.
                    mma_commit(bar(T::empty(stage)));
                }
                __syncwarp();
                issued = true;
                last_stage = stage;
                last_ph = ph;
                if (++stage == STAGES) { stage = 0; ph ^= 1u; }
                if (++tb == NBUF) { tb = 0; tph ^= 1u; }
            }
        }
        if (!ok && issued && lane == 0) drain_wait(bar(T::empty(last_stage)), last_ph, p0.timeout_ns);
        __syncwarp();
      } else if (warp == 2) {
        // ------------------------------------------------ scale loader
        int slot = 0;
        uint32_t sph = 0;
        bool ok = true;
        const uint32_t ring = sbase + T::OFF_SCALE;
        for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
            FP8BS_UNIT(u);
            int mb, nb;
            tile_coords(w.t, p, mb, nb);
            // One slot per K block (weight gradient) or per SBATCH K blocks.
            constexpr int step = SBMODE == SB_SCALAR ? T::SBATCH : 1;
            for (int kb = w.kb0; kb < w.kb1; kb += step) {
                if (!warp_wait_bounded(bar(T::sempty(slot)), sph ^ 1u, wc)) { ok = false; break; }
                const uint32_t dst = ring + static_cast<uint32_t>(slot * T::SLOT_FLOATS * 4);
                const float* sa_src = p.sa + static_cast<int64_t>(kb) * p.sa_ld + mb * BM;
                if constexpr (SBMODE == SB_SCALAR) {
                    // Row scales of blocks kb .. kb+n-1 at [j][128]; the weight scale
                    // of column half h of block kb+j at SBATCH*128 + 2j + h (a half past
                    // the output's last column block copies any valid scale: its
                    // results are never stored).
                    const int n = w.kb1 - kb < T::SBATCH ? w.kb1 - kb : T::SBATCH;
                    for (int j = 0; j < n; j++)
                        cp_async_16(dst + static_cast<uint32_t>(j * T::SA_FLOATS * 4 + lane * 16),
                                    sa_src + static_cast<int64_t>(j) * p.sa_ld + lane * 4);
                    if (lane < 2 * n) {
                        const int j = lane >> 1, h = lane & 1;
                        int jbh = (nb * BN + h * 128) >> 7;
                        if (jbh >= p.nb_valid) jbh = 0;
                        cp_async_4(dst + static_cast<uint32_t>((T::SBATCH * T::SA_FLOATS + 2 * j + h) * 4),
                                   p.sb + jbh * p.sb_stride_j + (kb + j) * p.sb_stride_b);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        // Row 32q + 8i' + u goes to 32q + 4u + i': the four rows a
                        // promotion thread holds (u = t/4) form one float4.
                        const int row = lane * 4 + i;
                        const int pos = (row & ~31) + 4 * (row & 7) + ((row >> 3) & 3);
                        cp_async_4(dst + pos * 4, sa_src + row);
                    }
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        // Column pair 2pr, 2pr+1 = h*128 + 64m + 8g + 2c + {0,1} goes to
                        // group (h, c) at 16m + 2g.  Columns past the output's end (a
                        // ragged last tile) copy any valid scale: they are never stored.
                        const int col = 2 * (lane * 4 + i);
                        const int h = col >> 7, w = col & 127;
                        const int pos = T::SA_FLOATS + h * T::SB_HALF + ((w >> 1) & 3) * T::SB_GROUP +
                                        16 * (w >> 6) + 2 * ((w >> 3) & 7);
                        int64_t gcol = static_cast<int64_t>(nb) * BN + col;
                        if (gcol >= p.cols) gcol = 0;
                        cp_async_8(dst + pos * 4, p.sb + static_cast<int64_t>(kb) * p.cols + gcol);
                    }
                }
                cp_async_arrive(bar(T::sfull(slot)));
                if (++slot == SSLOTS) { slot = 0; sph ^= 1u; }
            }
        }
        cp_async_wait_all();
      } else if constexpr (EPI == EPI_PLAIN) {
        // ------------------------------------------------ output store issuer
        // For the units whose plain BF16 epilogue it takes over (delegated_store),
        // waits until every promotion warp has staged its slice, issues the
        // tile's TMA stores, and frees the staging buffer once they have read
        // it, so that the promotion warps go on to the next tile at once.
        uint32_t oph = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
            FP8BS_UNIT(u);
            if (!delegated_store(p, w)) continue;
            int mb, nb;
            tile_coords(w.t, p, mb, nb);
            if (!uniform_wait(bar(T::ofull()), oph, wc)) { ok = false; break; }
            if (lane == 0) {
#pragma unroll 1
                for (int e = 0; e < NUM_EPI_WARPS; e++) {
                    const int q = e & 3, h = e >> 2;
                    const int32_t x0 = nb * BN + h * COLS, y0 = mb * BM + q * 32;
                    if ((x0 >> 7) >= p.nb_valid || static_cast<int64_t>(y0) >= p.rows) continue;
                    const uint32_t so = sbase + T::OFF_OUT + static_cast<uint32_t>(e * 2 * T::OUT_BOX_BYTES);
                    tma_store_2d(&grp.tmC[g], so, x0, y0);
                    tma_store_2d(&grp.tmC[g], so + T::OUT_BOX_BYTES, x0 + 64, y0);
                }
                bulk_commit_group();
                bulk_wait_read_all();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(T::ofree()));
            oph ^= 1u;
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(RegSplit<SBMODE>::epi));
        // ------------------------------------------------ promotion + epilogue
        const int ew = warp - 4;
        const int quad = warp & 3;   // TMEM lanes this warp may access
        const int half = ew >> 2;    // column half of the tile
        const int row = quad * 32 + lane;
        const float* ring = reinterpret_cast<const float*>(smem + T::OFF_SCALE);
        int tb = 0, slot = 0, stage = 0;
        uint32_t sph = 0, xph = 0, q8ph = 0, ph = 0;
        uint32_t delegated = 0;  // units whose stores warp 3 issued so far
        bool ok = true;
        for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
            FP8BS_UNIT(u);
            int mb, nb;
            tile_coords(w.t, p, mb, nb);
            // 128-column block of the output this warp's columns fall in
            const int jb = (nb * BN + half * COLS) >> 7;
            const bool jvalid = jb < p.nb_valid;
            float acc[COLS];
#pragma unroll
            for (int i = 0; i < COLS; i++) acc[i] = 0.0f;
            (void)jvalid;
            // Scale products sa * sb of the next K blocks of a batch (forward /
            // data gradient), shifted down one per block.
            float sc1 = 0.0f, sc2 = 0.0f, sc3 = 0.0f;
            static_assert(T::SBATCH == 4, "the batch is unpacked into sc1..sc3");
            for (int kb = w.kb0; kb < w.kb1; kb++) {
                const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) +
                                       static_cast<uint32_t>(tb * BN + half * COLS);
                uint32_t ra[32], rb[32];
                if constexpr (SBMODE == SB_SCALAR) {
                    // Accumulator slice in the .32x32b layout: thread = row, register =
                    // column; one scale per thread per K block.
                    float sc;
                    if (((kb - w.kb0) & (T::SBATCH - 1)) == 0) {
                        if (!uniform_wait(bar(T::sfull(slot)), sph, wc)) { ok = false; break; }
                        const float* sl = ring + slot * T::SLOT_FLOATS;
                        const float* sw2 = sl + T::SBATCH * T::SA_FLOATS + half;
                        const int n = w.kb1 - kb;
                        sc = __fmul_rn(sl[row], sw2[0]);
                        if (n > 1) sc1 = __fmul_rn(sl[T::SA_FLOATS + row], sw2[2]);
                        if (n > 2) sc2 = __fmul_rn(sl[2 * T::SA_FLOATS + row], sw2[4]);
                        if (n > 3) sc3 = __fmul_rn(sl[3 * T::SA_FLOATS + row], sw2[6]);
                        // The batch's scales are in registers: free the slot now.
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(T::sempty(slot)));
                        if (++slot == SSLOTS) { slot = 0; sph ^= 1u; }
                    } else {
                        sc = sc1;
                        sc1 = sc2;
                        sc2 = sc3;
                    }
                    if (!uniform_wait(bar(T::empty(stage)), ph, wc)) { ok = false; break; }
                    tc_fence_after();
                    // Two 32-column chunks in flight per wait; the TMEM buffer is
                    // released as soon as the last chunk is in registers.
                    tmem_ld_32cols(taddr + 0, ra);
                    tmem_ld_32cols(taddr + 32, rb);
                    tmem_wait_ld(ra);
                    reg_fence(rb);
                    promote_scalar(acc, 0, ra, sc);
                    promote_scalar(acc, 32, rb, sc);
                    tmem_ld_32cols(taddr + 64, ra);
                    tmem_ld_32cols(taddr + 96, rb);
                    tmem_wait_ld(ra);
                    reg_fence(rb);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(T::tempty(tb)));
                    promote_scalar(acc, 64, ra, sc);
                    promote_scalar(acc, 96, rb, sc);
                } else {
                    // Weight gradient: the scale is row scale x column scale, so the slice
                    // is read in the .16x256b layout (4 rows x 32 columns per thread), which
                    // needs 8 shared-memory loads of column scales per K block instead of
                    // 32 with one row per thread.  acc[32L + i]: L = 0,1 lanes 0-15 and
                    // L = 2,3 lanes 16-31 of the quadrant; L even columns 0-63, odd 64-127.
                    if (!warp_wait_bounded(bar(T::sfull(slot)), sph, wc)) { ok = false; break; }
                    const float* sl = ring + slot * T::SLOT_FLOATS;
                    const float4 sa4 = *reinterpret_cast<const float4*>(sl + quad * 32 + 4 * (lane >> 2));
                    const float* cs = sl + T::SA_FLOATS + half * T::SB_HALF + (lane & 3) * T::SB_GROUP;
                    if (!uniform_wait(bar(T::empty(stage)), ph, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t thi = taddr + (16u << 16);
                    tmem_ld_16x256b_x8(taddr, ra);
                    tmem_ld_16x256b_x8(thi, rb);
                    tmem_wait_ld(ra);
                    reg_fence(rb);
                    promote_rank1(acc, 0, 64, ra, rb, sa4, cs);
                    tmem_ld_16x256b_x8(taddr + 64, ra);
                    tmem_ld_16x256b_x8(thi + 64, rb);
                    tmem_wait_ld(ra);
                    reg_fence(rb);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(T::tempty(tb)));
                    promote_rank1(acc, 32, 96, ra, rb, sa4, cs + 16);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(T::sempty(slot)));
                    if (++slot == SSLOTS) { slot = 0; sph ^= 1u; }
                }
                if (++tb == NBUF) tb = 0;
                if (++stage == STAGES) { stage = 0; ph ^= 1u; }
            }
            if (!ok) break;
            if (w.split) {
                // Publish this warp's FP32 partial (lane-interleaved float4s, so
                // every store instruction writes 512 contiguous bytes), then count
                // it; the part that arrives last finishes the slice.
                const int64_t tile_id = w.t - p.tail_first;
                const float4* part0 = reinterpret_cast<const float4*>(p.ws) +
                                      (tile_id * p.splits * NUM_EPI_WARPS + ew) * 1024;
                float4* dst = reinterpret_cast<float4*>(p.ws) +
                              ((tile_id * p.splits + w.s) * NUM_EPI_WARPS + ew) * 1024;
#pragma unroll
                for (int c = 0; c < 32; c++)
                    dst[c * 32 + lane] = make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
                __threadfence();
                __syncwarp();
                uint32_t arrived = 0;
                if (lane == 0) arrived = count_arrival(p.arrivals + tile_id * NUM_EPI_WARPS + ew, p.epoch, wc);
                arrived = __shfl_sync(0xffffffffu, arrived, 0);
                if (arrived == 0u) { ok = false; break; }
                if (arrived != static_cast<uint32_t>(p.splits)) continue;
                // Last part: every partial is published.  Sum them in part order
                // (this part's own included, as published), whichever CTA this is.
                __threadfence();
#pragma unroll
                for (int c = 0; c < 32; c++) {
                    const float4 v = __ldcg(part0 + c * 32 + lane);
                    acc[4 * c] = v.x;
                    acc[4 * c + 1] = v.y;
                    acc[4 * c + 2] = v.z;
                    acc[4 * c + 3] = v.w;
                }
                for (int j = 1; j < p.splits; j++) {
                    const float4* src = part0 + static_cast<int64_t>(j) * NUM_EPI_WARPS * 1024;
#pragma unroll
                    for (int c = 0; c < 32; c++) {
                        const float4 v = __ldcg(src + c * 32 + lane);
                        acc[4 * c] += v.x;
                        acc[4 * c + 1] += v.y;
                        acc[4 * c + 2] += v.z;
                        acc[4 * c + 3] += v.w;
                    }
                }
            }
            if constexpr (SBMODE == SB_SCALAR) {
                if constexpr (EPI == EPI_SWIGLU) {
                    // SwiGLU: half 0 holds the gate values G of this 128-wide H block,
                    // half 1 the up values U of the same rows and columns.  The two
                    // warps of a quadrant share the activation: each hands the other,
                    // in the first box of its staging buffer (32 rows x 128 bytes,
                    // 16-byte chunk c of row r at c ^ (r % 8)), the BF16 half it needs
                    // -- the gate warp G[64..127], the up warp U[0..63] -- then the
                    // gate warp computes H[0..63] and the up warp H[64..127] and each
                    // stores its BF16 half.  The row's amax is combined through
                    // shared memory, and both FP8 halves are staged in the gate
                    // warp's first box for one TMA store.
                    const uint32_t own0 = sbase + T::OFF_OUT + static_cast<uint32_t>(ew * 2 * T::OUT_BOX_BYTES);
                    const uint32_t own1 = own0 + static_cast<uint32_t>(T::OUT_BOX_BYTES);
                    const uint32_t peer0 = sbase + T::OFF_OUT + static_cast<uint32_t>((ew ^ 4) * 2 * T::OUT_BOX_BYTES);
                    const uint32_t gate0 = sbase + T::OFF_OUT + static_cast<uint32_t>(quad * 2 * T::OUT_BOX_BYTES);
                    const int mine = half * 64;  // H columns this warp computes
                    // This warp's TMA stores of the previous tile have read its boxes.
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                    if (half == 0) stage_bf16_64<64>(acc, own0, lane);
                    else stage_bf16_64<0>(acc, own0, lane);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(T::xhalf(quad)));
                    if (!warp_wait_bounded(bar(T::xhalf(quad)), xph, wc)) { ok = false; break; }
                    float amax = half == 0 ? swiglu_64<0, true>(acc, peer0, lane) : swiglu_64<64, false>(acc, peer0, lane);
                    // Partial amax (a BF16 value) to the partner; both then hold the row's amax.
                    uint16_t* amx = reinterpret_cast<uint16_t*>(smem + T::OFF_AMAX);
                    amx[(quad * 2 + half) * 32 + lane] = static_cast<uint16_t>(__float_as_uint(amax) >> 16);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(T::xamax(quad)));
                    const bool hvalid = static_cast<int64_t>(mb) * BM + quad * 32 < p.rows;
                    if (hvalid && p.out_bf16) {
                        // This warp's 64 columns of H in BF16.
                        if (half == 0) stage_bf16_64<0>(acc, own1, lane);
                        else stage_bf16_64<64>(acc, own1, lane);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&grp.tmC[g], own1, nb * COLS + mine, mb * BM + quad * 32);
                            bulk_commit_group();
                        }
                    }
                    if (!warp_wait_bounded(bar(T::xamax(quad)), xph, wc)) { ok = false; break; }
                    xph ^= 1u;
                    amax = fmaxf(amax, __uint_as_float(static_cast<uint32_t>(amx[(quad * 2 + (half ^ 1)) * 32 + lane]) << 16));
                    float sq, inv;
                    tile_scale(amax, sq, inv);
                    if (half == 0) p.out_s[static_cast<int64_t>(nb) * p.sa_ld + static_cast<int64_t>(mb) * BM + row] = sq;
                    if (hvalid) {
                        // Both warps have read their handed-over halves (they published
                        // their amax after that), so the gate warp's first box is free
                        // for the FP8 row: chunks 0-3 from the gate warp, 4-7 from the up warp.
                        if (half == 0) stage_fp8_64<0, 0>(acc, inv, gate0, lane);
                        else stage_fp8_64<64, 4>(acc, inv, gate0, lane);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (half == 1) {
                            if (lane == 0) mbar_arrive(bar(T::xq8(quad)));
                        } else {
                            if (!warp_wait_bounded(bar(T::xq8(quad)), q8ph, wc)) { ok = false; break; }
                            if (lane == 0) {
                                tma_store_2d(&grp.tmQ[g], gate0, nb * COLS, mb * BM + quad * 32);
                                bulk_commit_group();
                            }
                        }
                        q8ph ^= 1u;
                    }
                    continue;
                }
            }
            // Output boxes that lie wholly past the last row (a token tail) are
            // not stored; TMA clips the rows of a partial box.
            const bool rvalid = static_cast<int64_t>(mb) * BM + quad * 32 < p.rows;
            // The staging buffer is free once warp 3's stores of the last
            // delegated unit have read it (the wait is satisfied at once when
            // they already have).
            if (delegated > 0 && !uniform_wait(bar(T::ofree()), (delegated - 1) & 1u, wc)) { ok = false; break; }
            if constexpr (EPI == EPI_PLAIN) {
                if (delegated_store(p, w)) {
                    const uint32_t stage_out = sbase + T::OFF_OUT + static_cast<uint32_t>(ew * 2 * T::OUT_BOX_BYTES);
                    if (jvalid && rvalid) {
                        stage_bf16_tile<SBMODE>(acc, stage_out, lane);
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(T::ofull()));
                    delegated++;
                    continue;
                }
            }
            if (jvalid && rvalid && p.out_f32_add) {
                // FP32 accumulate: four 32-row x 32-column boxes per warp, staged two
                // at a time (same 8 KB buffer, 128-byte swizzle: 16-byte chunk c of
                // row r at chunk c ^ (r % 8)) and added to global memory by TMA
                // reduce-add, so each output element receives exactly one FP32 add.
                const uint32_t stage_out = sbase + T::OFF_OUT + static_cast<uint32_t>(ew * 2 * T::OUT_BOX_BYTES);
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                    if constexpr (SBMODE == SB_SCALAR) {
#pragma unroll
                        for (int b = 0; b < 2; b++) {
#pragma unroll
                            for (int c = 0; c < 8; c++) {
                                const int j = h * 64 + b * 32 + c * 4;
                                const uint32_t a = stage_out + static_cast<uint32_t>(b * T::OUT_BOX_BYTES + lane * 128 +
                                                                                     ((c ^ (lane & 7)) << 4));
                                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(acc[j]),
                                             "f"(acc[j + 1]), "f"(acc[j + 2]), "f"(acc[j + 3])
                                             : "memory");
                            }
                        }
                    } else {
                        // .16x256b layout: columns 64h + 8g + 2(t%4) + {0,1} of rows
                        // 16Lh + t/4 + 8hi come from acc[32(h + 2Lh) + 4g + 2hi].
                        const int u = lane >> 2, c = lane & 3;
#pragma unroll
                        for (int lh = 0; lh < 2; lh++) {
#pragma unroll
                            for (int g = 0; g < 8; g++) {
#pragma unroll
                                for (int hi = 0; hi < 2; hi++) {
                                    const int j = 32 * (h + 2 * lh) + 4 * g + 2 * hi;
                                    const int rr = 16 * lh + 8 * hi + u;
                                    const int chunk = 2 * (g & 3) + (c >> 1);
                                    const uint32_t a = stage_out + static_cast<uint32_t>((g >> 2) * T::OUT_BOX_BYTES +
                                                                                         rr * 128 + ((chunk ^ u) << 4) +
                                                                                         8 * (c & 1));
                                    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(acc[j]), "f"(acc[j + 1])
                                                 : "memory");
                                }
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int32_t x0 = nb * BN + half * COLS + h * 64, y0 = mb * BM + quad * 32;
                        if (p.out_f32_add == 2) {
                            tma_store_2d(&grp.tmC[g], stage_out, x0, y0);
                            tma_store_2d(&grp.tmC[g], stage_out + T::OUT_BOX_BYTES, x0 + 32, y0);
                        } else {
                            tma_reduce_add_2d(&grp.tmC[g], stage_out, x0, y0);
                            tma_reduce_add_2d(&grp.tmC[g], stage_out + T::OUT_BOX_BYTES, x0 + 32, y0);
                        }
                        bulk_commit_group();
                    }
                }
            } else if (jvalid && rvalid && p.out_bf16) {
                // BF16 out through shared memory and two TMA stores (32 rows x 64
                // columns each) per warp.  The 128-byte swizzle puts the 16-byte
                // chunk c of row r at chunk c ^ (r % 8), so the 32 lanes' row
                // writes spread over all banks.
                const uint32_t stage_out = sbase + T::OFF_OUT + static_cast<uint32_t>(ew * 2 * T::OUT_BOX_BYTES);
                if (lane == 0) bulk_wait_read_all();  // the previous tile's stores have read the buffer
                __syncwarp();
                stage_bf16_tile<SBMODE>(acc, stage_out, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int32_t x0 = nb * BN + half * COLS, y0 = mb * BM + quad * 32;
                    tma_store_2d(&grp.tmC[g], stage_out, x0, y0);
                    tma_store_2d(&grp.tmC[g], stage_out + T::OUT_BOX_BYTES, x0 + 64, y0);
                    bulk_commit_group();
                }
            }
            if constexpr (SBMODE == SB_SCALAR) {
                if (EPI == EPI_FP8 && jvalid) {  // compile-time false outside the FP8 kernel
                    // FP8 output for the next linear: this thread holds one row's 128
                    // columns, i.e. one whole 1x128 tile.  Round to BF16 (the value the
                    // BF16 output holds), amax, the scheme's scale, E4M3 cast -- the
                    // operations of the row-wise quantizer on that BF16 row.
                    float amax = 0.0f;
#pragma unroll
                    for (int j = 0; j < COLS; j += 2) {
                        const uint32_t w2 = f32x2_to_bf16x2(acc[j], acc[j + 1]);
                        acc[j] = bf16lo_to_f32(w2);
                        acc[j + 1] = bf16hi_to_f32(w2);
                        amax = fmaxf(amax, fmaxf(fabsf(acc[j]), fabsf(acc[j + 1])));
                    }
                    float sq, inv;
                    tile_scale(amax, sq, inv);
                    // Scales of every row of the tile, padding rows (all-zero, s = 1) included.
                    p.out_s[static_cast<int64_t>(jb) * p.sa_ld + static_cast<int64_t>(mb) * BM + row] = sq;
                    if (rvalid) {
                        const uint32_t stage_out = sbase + T::OFF_OUT + static_cast<uint32_t>(ew * 2 * T::OUT_BOX_BYTES);
                        if (lane == 0) bulk_wait_read_all();  // earlier stores have read the buffer
                        __syncwarp();
#pragma unroll
                        for (int c = 0; c < 8; c++) {
                            uint32_t wv[4];
#pragma unroll
                            for (int q = 0; q < 4; q++) {
                                const int j = c * 16 + q * 4;
                                wv[q] = e4m3x2(__fmul_rn(acc[j], inv), __fmul_rn(acc[j + 1], inv)) |
                                        (e4m3x2(__fmul_rn(acc[j + 2], inv), __fmul_rn(acc[j + 3], inv)) << 16);
                            }
                            const uint32_t a = stage_out + static_cast<uint32_t>(lane * 128 + ((c ^ (lane & 7)) << 4));
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(wv[0]), "r"(wv[1]),
                                         "r"(wv[2]), "r"(wv[3])
                                         : "memory");
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&grp.tmQ[g], stage_out, nb * BN + half * COLS, mb * BM + quad * 32);
                            bulk_commit_group();
                        }
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

#undef FP8BS_UNIT
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace gemm
}  // namespace fp8bs
