// fp8bs.cu -- host side of the C ABI declared in include/fp8bs.h: argument
// validation, TMA tensor-map encoding (cached), split-K and tile-order
// planning for the GEMMs, kernel launches on the caller's stream, and the
// per-device status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "fp8bs.h"
#include "act.cuh"
#include "gemm.cuh"
#include "quant.cuh"

namespace fp8bs {

// Per-device status word written by kernels that give up a bounded wait.
__device__ uint32_t g_device_status;

// Scratch of fp8bs_gemm_wgrad_noalloc: split-K arrival counters (first 64 KiB) and FP32
// partial sums, in static device memory that exists on every device where
// this library's kernels are loaded, for the life of the process.  In host
// code this name is only a handle: its device address comes from
// cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[FP8BS_NOALLOC_SCRATCH_BYTES];

// Test hook: holds one SM per CTA (its shared memory leaves room for no
// other CTA of the library's GEMMs) for `ns` nanoseconds, then exits.
__global__ void occupy_kernel(int64_t ns) {
    extern __shared__ uint8_t held[];
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < static_cast<uint64_t>(ns)) __nanosleep(2000);
    if (threadIdx.x == 0) reinterpret_cast<volatile uint8_t*>(held)[0] = 0;
}
constexpr int kOccupySmem = 200 * 1024;

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kDefaultTimeoutNs = 2000000000LL;

std::atomic<int64_t> g_launches{0};
std::atomic<int64_t> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int> g_fault{0};
std::atomic<int> g_force_strip{0};  // test hook: tile-order strip width (0: chosen per shape)
std::atomic<unsigned> g_debug_flags{0};

struct DeviceInfo {
    bool ready = false;
    bool arch_ok = false;
    int sm_count = 0;
    int64_t l2_bytes = 0;
    uint32_t* status = nullptr;
    // Kernel attributes set once per variant: [scale mode][grouped][epilogue].
    std::atomic<bool> gemm_attr_set[2][2][3] = {};
    // Caller-registered scratch for split-K GEMMs (fp8bs_set_workspace).
    uint8_t* ws = nullptr;
    int64_t ws_bytes = 0;
    std::atomic<uint64_t> epoch{0};  // split-K launch tags (64-bit: never wraps)
    // fp8bs_gemm_wgrad_noalloc: device address of g_noalloc_scratch on this
    // device, looked up by that entry point's first call here.
    bool noalloc_ready = false;
    uint8_t* noalloc_scratch = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dim_ok(int64_t d) { return d > 0 && (d % 128) == 0 && d <= (int64_t(1) << 31); }
// Token counts may be any positive number; token-major arrays use them
// rounded up to whole 128-token blocks.
bool tokens_ok(int64_t m) { return m > 0 && m <= (int64_t(1) << 31) - 128; }
int64_t padded_tokens(int64_t m) { return (m + 127) / 128 * 128; }

// Looks up (once per device) whether this device can run the sm_103a
// kernels, its SM count and the device address of the status word.
int current_device(DeviceInfo** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return FP8BS_ERR_ARCH;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0, l2 = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
            cudaGetLastError();
            return FP8BS_ERR_ARCH;
        }
        d.l2_bytes = l2;
        d.arch_ok = (major == 10 && minor == 3);
        d.sm_count = sms;
        if (d.arch_ok) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) {
                cudaGetLastError();
                return FP8BS_ERR_LAUNCH;
            }
            d.status = static_cast<uint32_t*>(p);
        }
        d.ready = true;
    }
    if (!d.arch_ok) return FP8BS_ERR_ARCH;
    *out = &d;
    return FP8BS_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        cudaGetLastError();
    });
    return g_encode;
}

// Cache of encoded TMA tensor maps.  An encoded map is a pure function of
// its arguments (element type, base address, extents, row stride, box,
// swizzle), so a cached map is always the one the driver would encode
// again; the cache only saves the driver call on the launch path.
struct TmapKey {
    uint64_t base, inner, outer, row_bytes;
    uint32_t dt, box_inner, box_outer, sw;
    bool operator==(const TmapKey& o) const {
        return base == o.base && inner == o.inner && outer == o.outer && row_bytes == o.row_bytes && dt == o.dt &&
               box_inner == o.box_inner && box_outer == o.box_outer && sw == o.sw;
    }
};
struct TmapKeyHash {
    size_t operator()(const TmapKey& k) const {
        uint64_t h = 1469598103934665603ull;
        for (uint64_t v : {k.base, k.inner, k.outer, k.row_bytes, uint64_t(k.dt), uint64_t(k.box_inner),
                           uint64_t(k.box_outer), uint64_t(k.sw)}) {
            h ^= v;
            h *= 1099511628211ull;
        }
        return static_cast<size_t>(h);
    }
};
constexpr size_t kTmapCacheMax = 4096;  // entries; the cache is emptied when it fills
std::mutex g_tmap_mu;
std::unordered_map<TmapKey, CUtensorMap, TmapKeyHash> g_tmap_cache;
std::atomic<int64_t> g_tmap_encodes{0};

// 2-D row-major tensor [outer][inner] of `elem` bytes per element.
bool tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
             uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    const TmapKey key{reinterpret_cast<uint64_t>(base), inner, outer, row_bytes, static_cast<uint32_t>(dt),
                      box_inner, box_outer, static_cast<uint32_t>(sw)};
    {
        std::lock_guard<std::mutex> lk(g_tmap_mu);
        auto it = g_tmap_cache.find(key);
        if (it != g_tmap_cache.end()) {
            *m = it->second;
            return true;
        }
    }
    auto fn = encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    if (fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    g_tmap_encodes.fetch_add(1);
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    if (g_tmap_cache.size() >= kTmapCacheMax) g_tmap_cache.clear();
    g_tmap_cache.emplace(key, *m);
    return true;
}

int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FP8BS_OK : FP8BS_ERR_LAUNCH;
}

// Split-K plan: K splits of some output tiles so that the persistent
// launch's last wave is better filled.  Two forms:
//   uniform: every tile in S parts (S = 2..4, at least 16 K blocks each);
//   tail:    the tiles past the last full wave in S parts (S x tail tiles
//            <= SMs, at least 4 K blocks each), the full waves whole.
// Plans are compared by estimated time in K-block units (~0.6 us each): a
// unit adds one block for its set-up and store; the publication of a part's
// 128 KB FP32 partial costs ~5 blocks and the last part's read-and-add ~2
// blocks per partial (both limited by one SM's ~100 GB/s to L2, measured
// on B300).  A plan is used only if it saves at least 5% over no split, and
// only while its arrival counters fit the fixed counter region.  So short
// contractions (a forward product with K = 2048) are never split: moving
// the partials would cost more than the idle SMs of the last wave.
// Scratch layout: the counters ([split tiles][8 warps] x 8 bytes) in the
// first kFlagBytes, then one FP32 partial per part of every split tile.
constexpr int64_t kFlagBytes = 64 * 1024;         // counter region at the start of the scratch
constexpr int64_t kPartialBytes = 128 * 256 * 4;  // one tile's FP32 partial
struct SplitPlan {
    int splits;
    int64_t tail_first;  // tiles [0, tail_first) are not split
    int64_t units;
    int64_t bytes;       // scratch needed (0 without splitting)
};
SplitPlan plan_splits(int64_t tiles, int64_t kblocks, int sms) {
    auto waves = [&](int64_t units) { return static_cast<double>((units + sms - 1) / sms); };
    constexpr double kUnitCost = 1.0, kPublishCost = 5.0, kAddCost = 2.0;
    SplitPlan best{1, 0, tiles, 0};
    const double t_none = waves(tiles) * (static_cast<double>(kblocks) + kUnitCost);
    double best_t = t_none;
    auto consider = [&](int s, int64_t first, double t) {
        const int64_t split_tiles = tiles - first;
        if (split_tiles * gemm::NUM_EPI_WARPS * 8 > kFlagBytes) return;
        if (t < best_t && t <= 0.95 * t_none) {
            best = {s, first, first + s * split_tiles, kFlagBytes + s * split_tiles * kPartialBytes};
            best_t = t;
        }
    };
    for (int s = 2; s <= 4; s++) {
        if (kblocks / s < 16) continue;
        const double k = static_cast<double>((kblocks + s - 1) / s);
        consider(s, 0, waves(tiles * s) * (k + kUnitCost) + kPublishCost + kAddCost * s);
    }
    const int64_t full = (tiles / sms) * sms, tail = tiles - full;
    if (full > 0 && tail > 0) {
        for (int s = 2; s <= 8; s++) {
            if (s * tail > sms || kblocks / s < 4) continue;
            const double k = static_cast<double>((kblocks + s - 1) / s);
            consider(s, full, static_cast<double>(tiles / sms) * (static_cast<double>(kblocks) + kUnitCost) +
                                  (k + kUnitCost) + kPublishCost + kAddCost * s);
        }
    }
    return best;
}

// One product in the kernel's operand roles: C[rows][cols] = A[rows][kc] *
// B[cols][kc]^T with row scales sa [kc/128][padded rows] and B scales
// either scalar (sb[jb * sb_stride_j + b * sb_stride_b]) or per column
// (sb [kc/128][cols]).
struct GemmSpec {
    int sbmode;
    const uint8_t* A;
    const uint8_t* B;
    int64_t rows, cols, kc;
    const float* sa;
    const float* sb;
    int64_t sb_stride_j, sb_stride_b;
    void* out;             // BF16 (or FP32 with out_f32_add); may be null when out_q is set
    bool out_f32_add;
    bool out_f32_store = false;  // test mode: FP32 out = the unrounded accumulator
    uint8_t* out_q = nullptr;  // forward only: 1x128-quantized output and its scales
    float* out_s = nullptr;
    bool swiglu = false;       // forward of an interleaved gate+up weight: outputs are H = SiLU(gate) * up
};

// The operand roles of product `op` called with its entry point's arguments.
GemmSpec spec_of(int op, const uint8_t* a, const float* sa, const uint8_t* b, const float* sb, void* out,
                 int64_t M, int64_t N, int64_t K, bool out_f32_add = false) {
    switch (op) {
        case FP8BS_OP_FPROP:
            // A = Xq [M][K] (row scales sx [K/128][Mp]); B = Wq [N][K]; the B scale of
            // output column block jb and K block b is sw[jb][b].
            return {gemm::SB_SCALAR, a, b, M, N, K, sa, sb, K / 128, 1, out, false};
        case FP8BS_OP_DGRAD:
            // A = dYq [M][N] (row scales sdy [N/128][Mp]); B = WqT [K][N]; contraction
            // block b is a 128-row block of W, output column block jb a 128-column
            // block of W: scale sw[b][jb].
            return {gemm::SB_SCALAR, a, b, M, K, N, sa, sb, 1, K / 128, out, false};
        default:
            // A = dYTq [N][Mp] (row scales sdyT [Mp/128][N]); B = XTq [K][Mp] with a
            // per-column scale vector sxT [Mp/128][K].  Contraction over the tokens,
            // padded to whole 128-token blocks (the transposed quantizer writes zero
            // payloads for the padding).
            return {gemm::SB_VECTOR, a, b, N, K, padded_tokens(M), sa, sb, 0, 0, out, out_f32_add};
    }
}

// Tile order of the persistent schedule: column strips c tiles wide,
// row-major inside a strip (c = n_tiles: plain row-major).  The CTAs run
// about `grid` work units at a time (a "wave"); every unit streams the K
// range of one A panel (128 rows x kc bytes) and one B panel (256 rows x kc
// bytes).  A panel that a wave needs comes from L2 if it was last used
// recently enough -- the bytes touched since (the panels and outputs of the
// waves in between, and half of the two waves themselves) fit in 70% of L2
// -- and from DRAM otherwise.  raster_dram_bytes estimates the DRAM bytes of
// panels that order reads; the estimate lands within 3% of the reads ncu
// measured on the decoder-layer products at 32768 tokens, in row-major and in
// strip orders alike.
double raster_dram_bytes(int64_t m_tiles, int64_t n_tiles, int64_t kc, int64_t c, int32_t splits,
                         int64_t tail_first, int64_t grid, double budget, double out_tile_bytes) {
    const int64_t tiles = m_tiles * n_tiles;
    const int64_t whole = splits > 1 ? tail_first : tiles;
    const int64_t units = whole + (splits > 1 ? splits * (tiles - tail_first) : 0);
    const double pa = 128.0 * static_cast<double>(kc), pb = 256.0 * static_cast<double>(kc);
    std::vector<int64_t> last_a(static_cast<size_t>(m_tiles), -1), last_b(static_cast<size_t>(n_tiles), -1);
    std::vector<int64_t> seen_a(static_cast<size_t>(m_tiles), -1), seen_b(static_cast<size_t>(n_tiles), -1);
    std::vector<double> prefix(1, 0.0), ws_of;  // prefix[w]: working-set bytes of waves 0 .. w-1
    std::vector<int64_t> wave_a, wave_b;
    const int64_t per_strip = m_tiles * c;
    double reads = 0.0;
    for (int64_t w0 = 0, wi = 0; w0 < units; w0 += grid, wi++) {
        wave_a.clear();
        wave_b.clear();
        double out_bytes = 0.0;
        for (int64_t v = w0; v < std::min(units, w0 + grid); v++) {
            const int64_t t = v < whole ? v : tail_first + (v - whole) % (tiles - tail_first);
            const int64_t si = t / per_strip, loc = t - si * per_strip;
            const int64_t width = std::min(c, n_tiles - si * c);
            const size_t mb = static_cast<size_t>(loc / width), nb = static_cast<size_t>(si * c + loc % width);
            if (seen_a[mb] != wi) { seen_a[mb] = wi; wave_a.push_back(static_cast<int64_t>(mb)); }
            if (seen_b[nb] != wi) { seen_b[nb] = wi; wave_b.push_back(static_cast<int64_t>(nb)); }
            out_bytes += v < whole ? out_tile_bytes : 128.0 * 256.0 * 4.0;  // a split part writes FP32
        }
        const double ws = static_cast<double>(wave_a.size()) * pa + static_cast<double>(wave_b.size()) * pb + out_bytes;
        auto visit = [&](std::vector<int64_t>& last, int64_t i, double bytes) {
            const int64_t u = last[static_cast<size_t>(i)];
            const bool hit = u >= 0 && prefix[static_cast<size_t>(wi)] - prefix[static_cast<size_t>(u + 1)] +
                                               0.5 * (ws_of[static_cast<size_t>(u)] + ws) <= budget;
            if (!hit) reads += bytes;
            last[static_cast<size_t>(i)] = wi;
        };
        for (int64_t mb : wave_a) visit(last_a, mb, pa);
        for (int64_t nb : wave_b) visit(last_b, nb, pb);
        ws_of.push_back(ws);
        prefix.push_back(prefix.back() + ws);
    }
    return reads;
}

struct RasterKey {
    int64_t m_tiles, n_tiles, kc, tail_first, grid, l2;
    int32_t splits, out_bytes;
    bool operator==(const RasterKey& o) const {
        return m_tiles == o.m_tiles && n_tiles == o.n_tiles && kc == o.kc && tail_first == o.tail_first &&
               grid == o.grid && l2 == o.l2 && splits == o.splits && out_bytes == o.out_bytes;
    }
};
struct RasterKeyHash {
    size_t operator()(const RasterKey& k) const {
        uint64_t h = 1469598103934665603ull;
        for (int64_t v : {k.m_tiles, k.n_tiles, k.kc, k.tail_first, k.grid, k.l2, int64_t(k.splits), int64_t(k.out_bytes)})
            h = (h ^ static_cast<uint64_t>(v)) * 1099511628211ull;
        return static_cast<size_t>(h);
    }
};
std::mutex g_raster_mu;
std::unordered_map<RasterKey, int32_t, RasterKeyHash> g_raster_cache;
constexpr size_t kRasterCacheMax = 4096;

// The strip width with the fewest estimated DRAM bytes (row-major on a tie
// within 0.1%).  Candidates: row-major, then widths 1 .. 64 while the
// simulated units stay under ~16M (beyond that, row-major) and no order so
// far reads every panel just once.  Memoised per
// shape, plan and device.  Examples at 32768 tokens: the 32768 x 11264 x 2048
// forward product stays row-major (A read once and B kept in L2: 90 MB of
// panels; strips of 10 would re-read A once per strip, 359 MB); the 2048 x
// 5632 weight gradient goes column by column (its 8 MB panels cannot stay in
// L2 from one wave to the next, so the fewer distinct panels per wave the
// better: 403 MB against 629 MB row-major).
int32_t choose_strip(int64_t m_tiles, int64_t n_tiles, int64_t kc, int32_t splits, int64_t tail_first,
                     int64_t grid, int64_t l2_bytes, int32_t out_bytes) {
    const RasterKey key{m_tiles, n_tiles, kc, tail_first, grid, l2_bytes, splits, out_bytes};
    {
        std::lock_guard<std::mutex> lk(g_raster_mu);
        auto it = g_raster_cache.find(key);
        if (it != g_raster_cache.end()) return it->second;
    }
    const int64_t tiles = m_tiles * n_tiles;
    const int64_t units = splits > 1 ? tail_first + splits * (tiles - tail_first) : tiles;
    const double budget = 0.7 * static_cast<double>(l2_bytes);
    const double out_tile = 128.0 * 256.0 * out_bytes;
    // No order reads less than every panel once.
    const double floor_bytes = static_cast<double>(m_tiles) * 128.0 * static_cast<double>(kc) +
                               static_cast<double>(n_tiles) * 256.0 * static_cast<double>(kc);
    int64_t best_c = n_tiles;
    int64_t work = units;
    double best = raster_dram_bytes(m_tiles, n_tiles, kc, n_tiles, splits, tail_first, grid, budget, out_tile);
    for (int64_t c = 1; c < n_tiles && c <= 64 && work + units <= (int64_t(1) << 24) && best > floor_bytes * 1.001;
         c++) {
        work += units;
        const double r = raster_dram_bytes(m_tiles, n_tiles, kc, c, splits, tail_first, grid, budget, out_tile);
        if (r < best * 0.999) {
            best = r;
            best_c = c;
        }
    }
    std::lock_guard<std::mutex> lk(g_raster_mu);
    if (g_raster_cache.size() >= kRasterCacheMax) g_raster_cache.clear();
    g_raster_cache.emplace(key, static_cast<int32_t>(best_c));
    return static_cast<int32_t>(best_c);
}

// Sets member p's tile order for the work units it will run (after its split plan).
void set_raster(const DeviceInfo* d, gemm::Params* p, int64_t units) {
    const int forced = g_force_strip.load();
    if (forced > 0) {
        p->strip = std::min<int32_t>(forced, p->n_tiles);
        return;
    }
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(units, d->sm_count));
    const int32_t out_bytes = p->out_f32_add != 0 ? 4 : (p->out_bf16 ? 2 : 1);
    p->strip = choose_strip(p->m_tiles, p->n_tiles, static_cast<int64_t>(p->kblocks) * gemm::BK, p->splits,
                            p->tail_first, grid, d->l2_bytes, out_bytes);
}

// Tensor maps and kernel parameters of one product, not split.
int fill_member(DeviceInfo* d, const GemmSpec& s, CUtensorMap* tmA, CUtensorMap* tmB, CUtensorMap* tmC,
                CUtensorMap* tmQ, gemm::Params* p) {
    using namespace gemm;
    constexpr int BN = 256;
    // Without a BF16 output the store map is encoded on the FP8 payload and never used.
    const void* cbase = s.out != nullptr ? s.out : static_cast<const void*>(s.out_q);
    const int64_t ocols = s.swiglu ? s.cols / 2 : s.cols;  // columns of the stored output
    if (!tmap_2d(tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, s.A, s.kc, s.rows, s.kc, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tmap_2d(tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, s.B, s.kc, s.cols, s.kc, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !((s.out_f32_add || s.out_f32_store) ? tmap_2d(tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, cbase, ocols, s.rows, ocols * 4, 32, 32,
                                  CU_TENSOR_MAP_SWIZZLE_128B)
                        : tmap_2d(tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cbase, ocols, s.rows, ocols * 2, 64, 32,
                                  CU_TENSOR_MAP_SWIZZLE_128B)))
        return FP8BS_ERR_LAUNCH;
    if (s.out_q != nullptr &&
        !tmap_2d(tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, s.out_q, ocols, s.rows, ocols, 128, 32,
                 CU_TENSOR_MAP_SWIZZLE_128B))
        return FP8BS_ERR_LAUNCH;
    p->out_swiglu = s.swiglu ? 1 : 0;
    p->out_f32_add = s.out_f32_store ? 2 : (s.out_f32_add ? 1 : 0);
    p->out_bf16 = s.out != nullptr ? 1 : 0;
    p->out_q = s.out_q != nullptr ? 1 : 0;
    p->out_s = s.out_s;
    p->m_tiles = static_cast<int32_t>((s.rows + BM - 1) / BM);
    p->sa_ld = padded_tokens(s.rows);
    p->n_tiles = static_cast<int32_t>((s.cols + BN - 1) / BN);
    p->kblocks = static_cast<int32_t>(s.kc / BK);
    p->strip = p->n_tiles;  // row-major until set_raster sees the split plan
    p->nb_valid = static_cast<int32_t>(s.cols / 128);
    p->rows = s.rows;
    p->cols = s.cols;
    p->sa = s.sa;
    p->sb = s.sb;
    p->sb_stride_j = s.sb_stride_j;
    p->sb_stride_b = s.sb_stride_b;
    p->out = static_cast<uint16_t*>(s.out);
    p->status = d->status;
    p->timeout_ns = static_cast<uint64_t>(g_timeout_ns.load());
    p->fault = 0;
    p->splits = 1;
    p->tail_first = 0;
    p->ws = nullptr;
    p->arrivals = nullptr;
    p->epoch = 0;
    if (static_cast<int64_t>(p->m_tiles) * p->n_tiles > (int64_t(1) << 30)) return FP8BS_ERR_SHAPE;
    return FP8BS_OK;
}

template <int SBMODE, int G, int EPI = gemm::EPI_PLAIN>
int launch_group(DeviceInfo* d, const gemm::Group<G>& grp, cudaStream_t st) {
    using namespace gemm;
    using T = Tile<256>;
    const int64_t units = grp.first_unit[grp.count];
    if (units <= 0) return FP8BS_OK;
    const int grid = static_cast<int>(units < d->sm_count ? units : d->sm_count);
    auto kern = gemm_kernel<SBMODE, 256, G, EPI>;
    std::atomic<bool>& attr = d->gemm_attr_set[SBMODE][G > 1 ? 1 : 0][EPI];
    if (!attr.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (!attr.load(std::memory_order_relaxed)) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES) != cudaSuccess)
                return launch_status();
            attr.store(true, std::memory_order_release);
        }
    }
    kern<<<grid, THREADS, T::SMEM_BYTES, st>>>(grp);
    g_launches.fetch_add(1);
    return launch_status();
}

// Test mode (fp8bs_debug_set_flags): the plain products write their FP32
// accumulators instead of BF16.
GemmSpec with_debug_flags(GemmSpec s) {
    if (g_debug_flags.load() & FP8BS_DEBUG_F32_OUT) s.out_f32_store = true;
    return s;
}

// A tag for one split-K launch (never 0: counters start cleared).
uint64_t next_epoch(DeviceInfo* d) { return d->epoch.fetch_add(1) + 1; }

// Makes member `p` run split plan `sp` with its scratch at `base`.
void apply_split(gemm::Params* p, const SplitPlan& sp, uint8_t* base, uint64_t epoch) {
    p->splits = sp.splits;
    p->tail_first = static_cast<int32_t>(sp.tail_first);
    p->arrivals = reinterpret_cast<unsigned long long*>(base);
    p->ws = reinterpret_cast<float*>(base + kFlagBytes);
    p->epoch = epoch;
}

// One product, split along K when the registered scratch allows a plan that pays.
int run_gemm(const GemmSpec& s, cudaStream_t st) {
    using namespace gemm;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc != FP8BS_OK) return rc;
    Group<1> grp;
    Params& p = grp.p[0];
    rc = fill_member(d, s, &grp.tmA[0], &grp.tmB[0], &grp.tmC[0], &grp.tmQ[0], &p);
    if (rc != FP8BS_OK) return rc;
    p.fault = g_fault.exchange(0);
    const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    int64_t units = tiles;
    // The SwiGLU epilogue pairs two warps of one CTA, which split parts
    // finishing in different CTAs could not do: those products stay whole.
    if (d->ws != nullptr && !s.swiglu) {
        const SplitPlan sp = plan_splits(tiles, p.kblocks, d->sm_count);
        if (sp.splits > 1 && sp.bytes <= d->ws_bytes) {
            apply_split(&p, sp, d->ws, next_epoch(d));
            units = sp.units;
        }
    }
    set_raster(d, &p, units);
    grp.count = 1;
    grp.first_unit[0] = 0;
    grp.first_unit[1] = static_cast<int32_t>(units);
    if (s.sbmode == SB_VECTOR) return launch_group<SB_VECTOR, 1>(d, grp, st);
    if (s.swiglu) return launch_group<SB_SCALAR, 1, EPI_SWIGLU>(d, grp, st);
    if (s.out_q != nullptr) return launch_group<SB_SCALAR, 1, EPI_FP8>(d, grp, st);
    return launch_group<SB_SCALAR, 1>(d, grp, st);
}

}  // namespace
}  // namespace fp8bs

using namespace fp8bs;

extern "C" {

int fp8bs_quantize_act(const void* x, int64_t rows, int64_t cols, unsigned flags, uint8_t* q, float* s,
                       uint8_t* qT, float* sT, void* stream) {
    const bool row = (flags & FP8BS_ROWWISE) != 0, colt = (flags & FP8BS_COLWISE_T) != 0;
    if (!x || (flags & ~(FP8BS_ROWWISE | FP8BS_COLWISE_T)) || (!row && !colt)) return FP8BS_ERR_INVALID_ARG;
    if ((row && (!q || !s)) || (colt && (!qT || !sT))) return FP8BS_ERR_INVALID_ARG;
    if (!tokens_ok(rows) || !dim_ok(cols) || padded_tokens(rows) / 128 > 65535) return FP8BS_ERR_SHAPE;
    if (!aligned16(x) || (row && (!aligned16(q) || !aligned16(s))) || (colt && (!aligned16(qT) || !aligned16(sT))))
        return FP8BS_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc != FP8BS_OK) return rc;
    const int64_t ld = padded_tokens(rows);
    const dim3 grid(static_cast<unsigned>(cols / 128), static_cast<unsigned>(ld / 128));
    const auto* xw = static_cast<const uint32_t*>(x);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (row && colt)
        quant_tile_kernel<QM_ROW | QM_COLT><<<grid, 256, 0, st>>>(xw, rows, cols, ld, q, s, qT, sT);
    else if (row)
        quant_tile_kernel<QM_ROW><<<grid, 256, 0, st>>>(xw, rows, cols, ld, q, s, nullptr, nullptr);
    else
        quant_tile_kernel<QM_COLT><<<grid, 256, 0, st>>>(xw, rows, cols, ld, nullptr, nullptr, qT, sT);
    g_launches.fetch_add(1);
    return launch_status();
}

int fp8bs_quantize_weight(const void* w, int64_t n, int64_t k, uint8_t* q, uint8_t* qT, float* s, void* stream) {
    if (!w || !q || !s) return FP8BS_ERR_INVALID_ARG;
    if (!dim_ok(n) || !dim_ok(k) || n / 128 > 65535) return FP8BS_ERR_SHAPE;
    if (!aligned16(w) || !aligned16(q) || !aligned16(s) || (qT && !aligned16(qT))) return FP8BS_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc != FP8BS_OK) return rc;
    const dim3 grid(static_cast<unsigned>(k / 128), static_cast<unsigned>(n / 128));
    quant_tile_kernel<QM_BLOCK><<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint32_t*>(w), n, k, n, q, s, qT, nullptr);
    g_launches.fetch_add(1);
    return launch_status();
}

static int check_gemm_args(const void* a, const void* sa, const void* b, const void* sb, const void* out,
                           int64_t M, int64_t N, int64_t K) {
    if (!a || !sa || !b || !sb || !out) return FP8BS_ERR_INVALID_ARG;
    if (!tokens_ok(M) || !dim_ok(N) || !dim_ok(K)) return FP8BS_ERR_SHAPE;
    if (!aligned16(a) || !aligned16(sa) || !aligned16(b) || !aligned16(sb) || !aligned16(out)) return FP8BS_ERR_ALIGN;
    return FP8BS_OK;
}

int fp8bs_gemm_fprop(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw, void* y, int64_t M,
                     int64_t N, int64_t K, void* stream) {
    int rc = check_gemm_args(xq, sx, wq, sw, y, M, N, K);
    if (rc != FP8BS_OK) return rc;
    return run_gemm(with_debug_flags(spec_of(FP8BS_OP_FPROP, xq, sx, wq, sw, y, M, N, K)), static_cast<cudaStream_t>(stream));
}

int fp8bs_gemm_fprop_quant(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw, void* y,
                           uint8_t* yq, float* sy, int64_t M, int64_t N, int64_t K, void* stream) {
    int rc = check_gemm_args(xq, sx, wq, sw, yq, M, N, K);
    if (rc != FP8BS_OK) return rc;
    if (sy == nullptr) return FP8BS_ERR_INVALID_ARG;
    if (!aligned16(sy) || (y != nullptr && !aligned16(y))) return FP8BS_ERR_ALIGN;
    GemmSpec s = spec_of(FP8BS_OP_FPROP, xq, sx, wq, sw, y, M, N, K);
    s.out_q = yq;
    s.out_s = sy;
    return run_gemm(s, static_cast<cudaStream_t>(stream));
}

int fp8bs_gemm_fprop_swiglu_quant(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw, void* h,
                                  uint8_t* hq, float* sh, int64_t M, int64_t N2, int64_t K, void* stream) {
    int rc = check_gemm_args(xq, sx, wq, sw, hq, M, N2, K);
    if (rc != FP8BS_OK) return rc;
    if (sh == nullptr) return FP8BS_ERR_INVALID_ARG;
    if (N2 % 256 != 0) return FP8BS_ERR_SHAPE;
    if (!aligned16(sh) || (h != nullptr && !aligned16(h))) return FP8BS_ERR_ALIGN;
    GemmSpec s = spec_of(FP8BS_OP_FPROP, xq, sx, wq, sw, h, M, N2, K);
    s.out_q = hq;
    s.out_s = sh;
    s.swiglu = true;
    return run_gemm(s, static_cast<cudaStream_t>(stream));
}

int fp8bs_gemm_dgrad(const uint8_t* dyq, const float* sdy, const uint8_t* wqT, const float* sw, void* dx,
                     int64_t M, int64_t N, int64_t K, void* stream) {
    int rc = check_gemm_args(dyq, sdy, wqT, sw, dx, M, N, K);
    if (rc != FP8BS_OK) return rc;
    return run_gemm(with_debug_flags(spec_of(FP8BS_OP_DGRAD, dyq, sdy, wqT, sw, dx, M, N, K)), static_cast<cudaStream_t>(stream));
}

int fp8bs_gemm_wgrad(const uint8_t* dyTq, const float* sdyT, const uint8_t* xTq, const float* sxT, void* dw,
                     int64_t M, int64_t N, int64_t K, void* stream) {
    int rc = check_gemm_args(dyTq, sdyT, xTq, sxT, dw, M, N, K);
    if (rc != FP8BS_OK) return rc;
    return run_gemm(with_debug_flags(spec_of(FP8BS_OP_WGRAD, dyTq, sdyT, xTq, sxT, dw, M, N, K)), static_cast<cudaStream_t>(stream));
}

int fp8bs_gemm_wgrad_accumulate_f32(const uint8_t* dyTq, const float* sdyT, const uint8_t* xTq, const float* sxT,
                                    float* dw, int64_t M, int64_t N, int64_t K, void* stream) {
    int rc = check_gemm_args(dyTq, sdyT, xTq, sxT, dw, M, N, K);
    if (rc != FP8BS_OK) return rc;
    return run_gemm(spec_of(FP8BS_OP_WGRAD, dyTq, sdyT, xTq, sxT, dw, M, N, K, true),
                    static_cast<cudaStream_t>(stream));
}

int fp8bs_gemm_group(const fp8bs_gemm_args* gemms, int count, void* stream) {
    using namespace gemm;
    static_assert(kGroupMax == FP8BS_GROUP_MAX, "group size");
    static_assert(sizeof(Group<kGroupMax>) <= 4096, "kernel parameter space");
    if (gemms == nullptr || count < 1 || count > FP8BS_GROUP_MAX) return FP8BS_ERR_INVALID_ARG;
    int sbmode = -1;
    for (int i = 0; i < count; i++) {
        const fp8bs_gemm_args& a = gemms[i];
        if (a.op != FP8BS_OP_FPROP && a.op != FP8BS_OP_DGRAD && a.op != FP8BS_OP_WGRAD) return FP8BS_ERR_INVALID_ARG;
        const int rc = check_gemm_args(a.a, a.sa, a.b, a.sb, a.out, a.M, a.N, a.K);
        if (rc != FP8BS_OK) return rc;
        const int mode = a.op == FP8BS_OP_WGRAD ? SB_VECTOR : SB_SCALAR;
        if (sbmode >= 0 && mode != sbmode) return FP8BS_ERR_INVALID_ARG;
        sbmode = mode;
    }
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc != FP8BS_OK) return rc;
    Group<kGroupMax> grp;
    grp.count = count;
    grp.first_unit[0] = 0;
    // Each member may split as it would alone, in its own region of the
    // registered scratch (members that no longer fit stay whole).
    int64_t ws_used = 0;
    const uint64_t epoch = d->ws != nullptr ? next_epoch(d) : 0;
    for (int i = 0; i < count; i++) {
        const fp8bs_gemm_args& a = gemms[i];
        rc = fill_member(d, spec_of(a.op, a.a, a.sa, a.b, a.sb, a.out, a.M, a.N, a.K), &grp.tmA[i], &grp.tmB[i],
                         &grp.tmC[i], &grp.tmQ[i], &grp.p[i]);
        if (rc != FP8BS_OK) return rc;
        int64_t member_units = static_cast<int64_t>(grp.p[i].m_tiles) * grp.p[i].n_tiles;
        if (d->ws != nullptr) {
            const SplitPlan sp = plan_splits(member_units, grp.p[i].kblocks, d->sm_count);
            if (sp.splits > 1 && ws_used + sp.bytes <= d->ws_bytes) {
                apply_split(&grp.p[i], sp, d->ws + ws_used, epoch);
                ws_used += sp.bytes;
                member_units = sp.units;
            }
        }
        set_raster(d, &grp.p[i], member_units);
        const int64_t end = grp.first_unit[i] + member_units;
        if (end > (int64_t(1) << 30)) return FP8BS_ERR_SHAPE;
        grp.first_unit[i + 1] = static_cast<int32_t>(end);
    }
    for (int i = count; i < kGroupMax; i++) grp.first_unit[i + 1] = grp.first_unit[count];
    grp.p[0].fault = g_fault.exchange(0);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return sbmode == SB_VECTOR ? launch_group<SB_VECTOR, kGroupMax>(d, grp, st)
                               : launch_group<SB_SCALAR, kGroupMax>(d, grp, st);
}

int fp8bs_set_workspace(void* ws, int64_t bytes) {
    if (bytes < 0 || (ws == nullptr && bytes != 0) || (ws != nullptr && bytes < kFlagBytes))
        return FP8BS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return FP8BS_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc != FP8BS_OK) return rc;
    if (ws != nullptr && cudaMemset(ws, 0, kFlagBytes) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    d->ws = static_cast<uint8_t*>(ws);
    d->ws_bytes = bytes;
    d->epoch.store(0);
    return FP8BS_OK;
}

int64_t fp8bs_gemm_workspace_bytes(int op, int64_t M, int64_t N, int64_t K) {
    if (op != FP8BS_OP_FPROP && op != FP8BS_OP_DGRAD && op != FP8BS_OP_WGRAD) return -FP8BS_ERR_INVALID_ARG;
    if (!tokens_ok(M) || !dim_ok(N) || !dim_ok(K)) return -FP8BS_ERR_SHAPE;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc != FP8BS_OK) return -rc;
    // Output tiles (128 x 256) and contraction blocks of each product.
    int64_t rows, cols, kc;
    switch (op) {
        case FP8BS_OP_FPROP: rows = M; cols = N; kc = K; break;
        case FP8BS_OP_DGRAD: rows = M; cols = K; kc = N; break;
        case FP8BS_OP_WGRAD: rows = N; cols = K; kc = padded_tokens(M); break;
        default: return -FP8BS_ERR_INVALID_ARG;
    }
    const int64_t tiles = ((rows + gemm::BM - 1) / gemm::BM) * ((cols + 255) / 256);
    return plan_splits(tiles, kc / gemm::BK, d->sm_count).bytes;
}

int64_t fp8bs_gemm_wgrad_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    return fp8bs_gemm_workspace_bytes(FP8BS_OP_WGRAD, M, N, K);
}

int fp8bs_gemm_wgrad_noalloc(const uint8_t* dyTq, const float* sdyT, const uint8_t* xTq, const float* sxT,
                             void* dw, int64_t M, int64_t N, int64_t K, void* stream) {
    using namespace gemm;
    int rc = check_gemm_args(dyTq, sdyT, xTq, sxT, dw, M, N, K);
    if (rc != FP8BS_OK) return rc;
    DeviceInfo* d = nullptr;
    rc = current_device(&d);
    if (rc != FP8BS_OK) return rc;
    {
        // Set-up, once per device, with that device current: the device
        // address of the static scratch.
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (!d->noalloc_ready) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
                cudaGetLastError();
                return FP8BS_ERR_CUDA;
            }
            d->noalloc_scratch = static_cast<uint8_t*>(ptr);
            d->noalloc_ready = true;
        }
    }
    // Same operand roles as fp8bs_gemm_wgrad: rows = N, cols = K, contraction M.
    const int64_t rows = N, cols = K, kc = padded_tokens(M);
    const int64_t tiles = (rows / BM) * ((cols + 255) / 256);
    if (tiles > (int64_t(1) << 30)) return FP8BS_ERR_SHAPE;
    const SplitPlan sp = plan_splits(tiles, kc / BK, d->sm_count);
    if (sp.bytes > static_cast<int64_t>(FP8BS_NOALLOC_SCRATCH_BYTES)) return FP8BS_ERR_SHAPE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Group<1> grp;
    Params& p = grp.p[0];
    rc = fill_member(d, spec_of(FP8BS_OP_WGRAD, dyTq, sdyT, xTq, sxT, dw, M, N, K), &grp.tmA[0], &grp.tmB[0],
                     &grp.tmC[0], &grp.tmQ[0], &p);
    if (rc != FP8BS_OK) return rc;
    if (sp.splits > 1) {
        // The array keeps whatever the previous call left; the arrival
        // counters carry this call's own tag, so nothing needs clearing
        // (partials are always written before they are read).
        apply_split(&p, sp, d->noalloc_scratch, next_epoch(d));
    }
    set_raster(d, &p, sp.units);
    grp.count = 1;
    grp.first_unit[0] = 0;
    grp.first_unit[1] = static_cast<int32_t>(sp.units);
    return launch_group<SB_VECTOR, 1>(d, grp, st);
}

int fp8bs_get_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc != FP8BS_OK) return rc;
    uint32_t v = 0, zero = 0;
    if (cudaMemcpy(&v, d->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    return (v & kStatusTimeout) ? FP8BS_ERR_TIMEOUT : FP8BS_OK;
}

const char* fp8bs_status_string(int status) {
    switch (status) {
        case FP8BS_OK: return "FP8BS_OK";
        case FP8BS_ERR_INVALID_ARG: return "FP8BS_ERR_INVALID_ARG";
        case FP8BS_ERR_SHAPE: return "FP8BS_ERR_SHAPE";
        case FP8BS_ERR_ALIGN: return "FP8BS_ERR_ALIGN";
        case FP8BS_ERR_ARCH: return "FP8BS_ERR_ARCH";
        case FP8BS_ERR_LAUNCH: return "FP8BS_ERR_LAUNCH";
        case FP8BS_ERR_TIMEOUT: return "FP8BS_ERR_TIMEOUT";
        case FP8BS_ERR_CUDA: return "FP8BS_ERR_CUDA";
        default: return "FP8BS_ERR_UNKNOWN";
    }
}

int64_t fp8bs_launch_count(void) { return g_launches.load(); }

int64_t fp8bs_debug_tensor_map_encodes(void) { return g_tmap_encodes.load(); }

int fp8bs_debug_set_wait_timeout_ns(int64_t ns) {
    if (ns < 0) return FP8BS_ERR_INVALID_ARG;
    g_timeout_ns.store(ns == 0 ? kDefaultTimeoutNs : ns);
    return FP8BS_OK;
}

int fp8bs_debug_split_plan(int64_t tiles, int64_t kblocks, int sms, int64_t* out) {
    using namespace fp8bs;
    if (tiles <= 0 || kblocks <= 0 || sms <= 0 || out == nullptr || tiles > (int64_t(1) << 30))
        return FP8BS_ERR_INVALID_ARG;
    const SplitPlan sp = plan_splits(tiles, kblocks, sms);
    out[0] = sp.splits;
    out[1] = sp.tail_first;
    out[2] = sp.units;
    out[3] = sp.bytes;
    return FP8BS_OK;
}

int fp8bs_debug_tile_order(int64_t m_tiles, int64_t n_tiles, int64_t kc, int32_t splits, int64_t tail_first,
                           int64_t grid, int64_t l2_bytes, int32_t out_bytes, int64_t* out) {
    using namespace fp8bs;
    if (m_tiles <= 0 || n_tiles <= 0 || kc <= 0 || grid <= 0 || l2_bytes <= 0 || out == nullptr ||
        m_tiles * n_tiles > (int64_t(1) << 30) || splits < 1 || (out_bytes != 1 && out_bytes != 2 && out_bytes != 4))
        return FP8BS_ERR_INVALID_ARG;
    if (splits > 1 && (tail_first < 0 || tail_first >= m_tiles * n_tiles)) return FP8BS_ERR_INVALID_ARG;
    const int32_t c = choose_strip(m_tiles, n_tiles, kc, splits, tail_first, grid, l2_bytes, out_bytes);
    const double budget = 0.7 * static_cast<double>(l2_bytes), out_tile = 128.0 * 256.0 * out_bytes;
    out[0] = c;
    out[1] = static_cast<int64_t>(raster_dram_bytes(m_tiles, n_tiles, kc, c, splits, tail_first, grid, budget, out_tile));
    out[2] = static_cast<int64_t>(
        raster_dram_bytes(m_tiles, n_tiles, kc, n_tiles, splits, tail_first, grid, budget, out_tile));
    return FP8BS_OK;
}

int fp8bs_debug_occupy_sms(int ctas, int64_t ns, void* stream) {
    if (ctas < 1 || ns < 0 || ns > 2000000000LL) return FP8BS_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc != FP8BS_OK) return rc;
    if (ctas > d->sm_count) return FP8BS_ERR_INVALID_ARG;
    if (cudaFuncSetAttribute(occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kOccupySmem) != cudaSuccess)
        return launch_status();
    occupy_kernel<<<ctas, 32, kOccupySmem, static_cast<cudaStream_t>(stream)>>>(ns);
    g_launches.fetch_add(1);
    return launch_status();
}

int fp8bs_debug_set_flags(unsigned flags) {
    if (flags & ~static_cast<unsigned>(FP8BS_DEBUG_F32_OUT)) return FP8BS_ERR_INVALID_ARG;
    g_debug_flags.store(flags);
    return FP8BS_OK;
}

int fp8bs_debug_force_tile_order(int strip) {
    if (strip < 0) return FP8BS_ERR_INVALID_ARG;
    fp8bs::g_force_strip.store(strip);
    return FP8BS_OK;
}

int fp8bs_debug_set_fault(int mode) {
    if (mode != 0 && mode != 1) return FP8BS_ERR_INVALID_ARG;
    g_fault.store(mode);
    return FP8BS_OK;
}

int fp8bs_debug_e4m3_encode_bits(uint32_t first, int64_t n, uint8_t* out, void* stream) {
    if (!out || n < 0) return FP8BS_ERR_INVALID_ARG;
    if (n > (int64_t(1) << 32) || static_cast<uint64_t>(first) + static_cast<uint64_t>(n) > (uint64_t(1) << 32))
        return FP8BS_ERR_SHAPE;
    if (!aligned16(out)) return FP8BS_ERR_ALIGN;
    if (n == 0) return FP8BS_OK;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc != FP8BS_OK) return rc;
    const int64_t groups = (n + 3) / 4;
    const int64_t want = (groups + 255) / 256;
    const int grid = static_cast<int>(want < 8 * d->sm_count ? want : 8 * d->sm_count);
    e4m3_encode_bits_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(first, n, out);
    g_launches.fetch_add(1);
    return launch_status();
}

int fp8bs_debug_silu_mul(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* h, void* stream) {
    if (!g || !u || !h || n < 0) return FP8BS_ERR_INVALID_ARG;
    if (n == 0) return FP8BS_OK;
    DeviceInfo* d = nullptr;
    int rc = current_device(&d);
    if (rc != FP8BS_OK) return rc;
    const int64_t want = (n + 255) / 256;
    const int grid = static_cast<int>(want < 8 * d->sm_count ? want : 8 * d->sm_count);
    silu_mul_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(g, u, n, h);
    g_launches.fetch_add(1);
    return launch_status();
}

}  // extern "C"
