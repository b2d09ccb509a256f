// Host side of the C ABI declared in include/gemm_tn_f16.h: argument checks,
// kernel planning, scratch memory, TMA tensor maps and launches.
//
// The operation is the TN GEMM D = alpha * A . B^T + beta * C of the
// "gemm_device 逐行解析" page (section 1, the kernel signature with alpha and
// beta; section 3, the axpby epilogue), with the (M,K)/(N,K) K-contiguous
// operand views of "cute(8) smem_gemm" (section 代码实现).  Unlike the pages'
// host code (torch::Tensor arguments, CUDA_CHECK calling exit() on failure),
// this layer takes plain pointers, never exits, and reports every failure as
// a gemm_status_t.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <limits>
#include <mutex>
#include <vector>

#include "gemm_tn_f16.h"
#include "internal.h"

namespace gtn {

// Device error word written by timed-out waits (see tc_gemm.cuh).
__device__ uint32_t g_error_word = 0;

// Device address of the error word on the current device (no allocation).
cudaError_t error_word_address(uint32_t** out) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_error_word);
    if (e == cudaSuccess) *out = static_cast<uint32_t*>(p);
    return e;
}

namespace {

thread_local int t_last_cuda_error = 0;

std::atomic<int64_t> g_opt_timeout_ns{2000000000ll};
std::atomic<int64_t> g_opt_skip_first_load{0};
std::atomic<int64_t> g_opt_force_bn{0};
std::atomic<int64_t> g_opt_force_pair{0};
std::atomic<int64_t> g_opt_force_splits{0};
std::atomic<int64_t> g_opt_force_swap{0};
std::atomic<int64_t> g_opt_force_generic{0};
std::atomic<int64_t> g_opt_force_pack{0};
std::atomic<int64_t> g_opt_stream_k{0};
std::atomic<int64_t> g_opt_group_m{0};
std::atomic<int64_t> g_opt_serpentine{0};
std::atomic<int64_t> g_opt_row_loader{0};
std::atomic<int64_t> g_opt_check_trim_d{0};
std::atomic<int64_t> g_opt_k_cluster{0};
std::atomic<int64_t> g_opt_small{0};

gemm_status_t cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return GEMM_ERR_CUDA;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// A fresh 56-bit tag for each stream-K launch: splitmix64 of a process-wide
// sequence number (a bijection, so no two launches share a tag), never zero.
unsigned long long next_sk_epoch() {
    static std::atomic<unsigned long long> seq{0};
    unsigned long long z = seq.fetch_add(1) + 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    z ^= z >> 31;
    z &= (1ull << 56) - 1;
    return z == 0 ? 1 : z;
}
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// ------------------------------------------------------------------ per-device state

struct DeviceState {
    bool ready = false;
    int sms = 0;
    int major = 0, minor = 0;
    uint32_t* err = nullptr;
    cudaMemPool_t pool = nullptr;
    int64_t capacity[kMaxVariants];  // resident CTAs per variant, 0 = not queried yet
    cudaStream_t copy_in = nullptr;   // host -> device copies of gemm_tn_f16_host
    cudaStream_t copy_out = nullptr;  // device -> host copies of gemm_tn_f16_host
};

constexpr int kMaxDevices = 64;
DeviceState g_devices[kMaxDevices];
std::mutex g_dev_mu;

gemm_status_t device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceState& d = g_devices[dev];
    if (!d.ready) {
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return cuda_fail(e);
        if (!(d.major == 10 && d.minor == 3)) return GEMM_ERR_UNSUPPORTED;  // kernels are built for sm_103a only
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_error_word)) != cudaSuccess) return cuda_fail(e);
        d.err = static_cast<uint32_t*>(p);
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if ((e = cudaMemPoolCreate(&d.pool, &props)) != cudaSuccess) return cuda_fail(e);
        uint64_t keep = UINT64_MAX;  // keep freed scratch cached in the pool
        if ((e = cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess)
            return cuda_fail(e);
        for (int64_t& c : d.capacity) c = 0;
        d.ready = true;
    }
    *out = &d;
    return GEMM_OK;
}

// ------------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// A few recently encoded maps per host thread: steady-state callers that reuse
// the same buffers skip the driver call (a map depends only on these fields).
struct MapCacheEntry {
    const void* base;
    int64_t inner, rows, batch, ld, stride;
    bool batched;
    uint32_t box_inner, box_rows;
    uint64_t stamp;
    CUtensorMap map;
};
constexpr int kMapCache = 16;
thread_local MapCacheEntry t_map_cache[kMapCache] = {};
thread_local uint64_t t_map_clock = 0;

bool encode_map_uncached(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t batch, int64_t ld,
                         int64_t stride, bool batched, uint32_t box_inner, uint32_t box_rows);

// 3-D fp16 tensor map over (inner, rows, batch) with a box of (box_inner, box_rows, 1)
// and 128-byte swizzle.  `batched` false maps a single matrix (batch extent 1).
bool encode_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t batch, int64_t ld,
                int64_t stride, bool batched, uint32_t box_inner, uint32_t box_rows) {
    const uint64_t now = ++t_map_clock;
    int victim = 0;
    for (int i = 0; i < kMapCache; ++i) {
        MapCacheEntry& e = t_map_cache[i];
        if (e.stamp != 0 && e.base == base && e.inner == inner && e.rows == rows && e.batch == batch && e.ld == ld &&
            e.stride == stride && e.batched == batched && e.box_inner == box_inner && e.box_rows == box_rows) {
            e.stamp = now;
            *map = e.map;
            return true;
        }
        if (e.stamp < t_map_cache[victim].stamp) victim = i;
    }
    if (!encode_map_uncached(map, base, inner, rows, batch, ld, stride, batched, box_inner, box_rows)) return false;
    t_map_cache[victim] = {base, inner, rows, batch, ld, stride, batched, box_inner, box_rows, now, *map};
    return true;
}

bool encode_map_uncached(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t batch, int64_t ld,
                         int64_t stride, bool batched, uint32_t box_inner, uint32_t box_rows) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(batched ? batch : 1)};
    const int64_t st = batched ? stride : ld * rows;
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2u, static_cast<cuuint64_t>(st) * 2u};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// fp32 split-K partials W[slice][M][N] (slices = batch x splits) for TMA stores: boxes of
// 32 rows x 32 columns (128 bytes) with 128-byte swizzle.  Needs N % 4 == 0.
bool encode_partials_map(CUtensorMap* map, const float* W, int64_t M, int64_t N, int64_t slices) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn || N % 4 != 0) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(slices)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 4u, static_cast<cuuint64_t>(M * N) * 4u};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(W), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ problem + plan

struct Problem {
    int64_t M, N, K, batch;
    int64_t lda, ldb, ldc, ldd;
    int64_t sA, sB, sC, sD;
    float beta;
    uint32_t align;  // bit i: operand i (A,B,C,D) base is 16-byte aligned
    int32_t a_mn = 0, b_mn = 0;  // 1: A stored K x lda (M contiguous) / B stored K x ldb (N contiguous)
    int32_t acc16 = 0;           // 1: accumulate in fp16 on the tensor core
};

// Elements of an operand's rows in memory (its contiguous extent) and their count.
int64_t a_rows(const Problem& p) { return p.a_mn ? p.K : p.M; }
int64_t a_len(const Problem& p) { return p.a_mn ? p.M : p.K; }
int64_t b_rows(const Problem& p) { return p.b_mn ? p.K : p.N; }
int64_t b_len(const Problem& p) { return p.b_mn ? p.N : p.K; }

struct Plan {
    gemm_tn_plan_t pub;
    TcVariant var;
    int32_t epi;
    int64_t rows_a, rows_b;
    int64_t tiles_m, tiles_n;
    int64_t ldo_a, ldo_b;        // leading dims of the packed copies
    int64_t pack_a_bytes, pack_b_bytes, partial_bytes;
    int64_t sk_w_bytes, sk_ctr_bytes;  // stream-K partial slots and arrival counters
    int64_t sk_iters;
    int group_m;
    int32_t rl, rl_a, rl_b;  // row-loader variant; A / B read by its loader warps (not repacked)
    int32_t ck;              // cluster K split: the two CTAs of a cluster take the two halves of K
    int32_t small_bn;        // > 0: small-problem kernel with tiles of 128 x small_bn
};

bool operand_tma_ok(bool aligned16, int64_t ld, int64_t stride, int64_t batch) {
    return aligned16 && ld % 8 == 0 && (batch == 1 || stride % 8 == 0);
}

gemm_status_t validate(const Problem& p) {
    if (p.M < 0 || p.N < 0 || p.K < 0 || p.batch < 0) return GEMM_ERR_INVALID_VALUE;
    const int64_t lim = int64_t(1) << 31;
    if (p.M >= lim || p.N >= lim || p.K >= lim || p.batch >= lim) return GEMM_ERR_UNSUPPORTED;
    if (p.M == 0 || p.N == 0 || p.batch == 0) return GEMM_OK;
    if (p.ldd < std::max<int64_t>(p.N, 1)) return GEMM_ERR_INVALID_VALUE;
    if (p.K > 0 && (p.lda < a_len(p) || p.ldb < b_len(p))) return GEMM_ERR_INVALID_VALUE;
    if (p.beta != 0.0f && p.ldc < std::max<int64_t>(p.N, 1)) return GEMM_ERR_INVALID_VALUE;
    if (p.batch > 1) {
        if (p.sA < 0 || p.sB < 0 || p.sC < 0 || p.sD < 0) return GEMM_ERR_INVALID_VALUE;
        if (p.sD < (p.M - 1) * p.ldd + p.N) return GEMM_ERR_INVALID_VALUE;  // output entries must be disjoint
    }
    return GEMM_OK;
}

// Stream-K split of the tiles over `groups` CTA groups (host arithmetic only).
// The tiles that fill whole waves run data-parallel; when the last wave would
// leave groups idle, its tiles' k-blocks are spread over every group instead.
void plan_stream_k(const Problem& pr, Plan& pl, int64_t groups) {
    gemm_tn_plan_t& pub = pl.pub;
    const int pair = pub.cta_pair;
    const int64_t tiles = pl.tiles_m * pl.tiles_n * pr.batch;
    const int64_t kb = ceil_div(pr.K, 64);
    const int64_t G = std::max<int64_t>(groups, 1);
    pub.stream_k = 0;
    pub.sk_maxc = 0;
    pub.dp_tiles = tiles;
    pub.sk_tiles = 0;
    pl.sk_iters = 0;
    pl.sk_w_bytes = pl.sk_ctr_bytes = 0;
    const bool sk_epi = pl.epi == EPI_TMA || pl.epi == EPI_TMA_C || pl.epi == EPI_TMA_CG || pl.epi == EPI_VEC ||
                        pl.epi == EPI_GENERIC || pl.epi == EPI_SWAP;
    // Stream-K trades the idle part of the last wave for fix-up work: every contributor
    // to a split tile parks its fp32 partial (128 x tile_n per CTA) and the last one sums
    // them and runs the epilogue, holding up its own later tiles meanwhile.  Measured on
    // GB300 (data-parallel against stream-K), it pays only when the saved share of a wave
    // is long or the partials are small:
    //   - narrow swapped tiles (tile_n <= 32): 16x8192x8192 33.9 against 43.2 us;
    //   - 128 or more k-blocks per tile: 2560^2x8192 67.9 against 82.2 us, 4096^2x8192
    //     155 against 166 us (one loss, 256x8192x8192, where both sides are bound by
    //     reading B: 65.7 against 59.6 us);
    //   - 64 k-blocks per tile behind at least three whole waves, which hide the fix-ups:
    //     4096^3 85.1 against 86.3 us, 5120^2x4096 124.8 against 128.0 us;
    // and in each case the idle part of the last wave is worth at least 36 k-blocks
    // (8192^3, last wave 47 % full: 586.9 against 597.0 us; 4096x8192x4096, 17 k-blocks:
    // 154.8 against 150.1 us).  Shorter K, fewer waves, a small saving or many
    // contributors per split tile lose, often badly: 2048^2x1024 32.9 against 14.3 us,
    // 1280x4096x4096 (19 contributors per split tile) 99.9 against 47.1 us,
    // 384x4096x4096 38.5 against 32.8 us.  Forced on, stream-K applies whenever the
    // tiles do not divide evenly.
    const int64_t mode = g_opt_stream_k.load();
    int64_t sk_groups = 0;  // CTA groups of a stream-K launch
    if (mode >= 0 && sk_epi && pub.splits == 1 && kb >= 8 && tiles % G != 0) {
        // k-blocks a group would idle through in the last data-parallel wave
        const double saved_kb = static_cast<double>(ceil_div(tiles, G) * G - tiles) / static_cast<double>(G) *
                                static_cast<double>(kb);
        // Every group must get at least one iteration (contributors to a tile are
        // then consecutive groups); with no whole wave, launch fewer groups instead.
        int64_t Gs = G;
        if (tiles < G) Gs = std::min(G, tiles * kb);
        // Long K on a few tiles (operand layouts without a split-K variant): data-parallel
        // would leave most of the GPU idle for a long time, so split anyway, over at most
        // 16 groups per tile (the fix-up reads every contributor's partial in turn; 26
        // per tile measured slower, 256 x 384 x 131072: 100 against 65 us).
        const bool long_k = mode == 0 && kb >= 128 && tiles * 4 <= G;
        if (long_k) Gs = std::min<int64_t>(Gs, tiles * 16);
        const int64_t dp = (tiles / Gs) * Gs;
        const int64_t sk = tiles - dp;
        const int64_t I = sk * kb;
        TcVariant skv;
        if (I >= Gs && find_tc_variant(pl.var.bn, pl.var.pair, pl.epi | (pl.rl ? EPI_RL : 0) | (pl.ck ? EPI_CK : 0), 1,
                                       &skv)) {
            auto owner = [&](int64_t i) { return ((i + 1) * Gs - 1) / I; };
            int64_t maxc = 1;
            for (int64_t t = 0; t < sk; ++t) maxc = std::max(maxc, owner((t + 1) * kb - 1) - owner(t * kb) + 1);
            const bool narrow = pub.tile_n <= 32;
            const bool pays = narrow || long_k ||
                              (pub.tile_n <= 256 && maxc <= 8 && saved_kb >= 36.0 &&
                               (kb >= 128 || (kb >= 64 && tiles >= 3 * G)));
            if (mode > 0 || pays) {
                pub.stream_k = 1;
                pub.sk_maxc = static_cast<int32_t>(maxc);
                pub.dp_tiles = dp;
                pub.sk_tiles = sk;
                pl.sk_iters = I;
                pl.sk_w_bytes = round_up(sk * maxc * pair * 128 * static_cast<int64_t>(pub.tile_n) * 4, 256);
                pl.sk_ctr_bytes = round_up(sk * pair * 4 * 8, 256);
                sk_groups = Gs;
            }
        }
    }
    find_tc_variant(pl.var.bn, pl.var.pair, pl.epi | (pl.rl ? EPI_RL : 0) | (pl.ck ? EPI_CK : 0), pub.stream_k,
                    &pl.var);
    // Wide data-parallel tiles with D = alpha*acc by TMA stores: the variant with one epilogue
    // warpgroup per part of the accumulator, which hands both parts back to the MMA as soon
    // as they are in registers (the next tile's MMAs otherwise wait for the stores of the
    // first part before they get the second).
    TcVariant h2v;
    if (!pub.stream_k && !pl.rl && !pl.ck && pl.var.bn > 256 && pl.epi == EPI_TMA &&
        find_tc_variant(pl.var.bn, pl.var.pair, EPI_TMA | EPI_H2, 0, &h2v))
        pl.var = h2v;
    // Tiles of a single k-block (K <= 64: the attention score Q K^T) spend their time storing
    // D: the variant with four staging buffers per epilogue warp and a three-stage ring keeps
    // more TMA stores in flight (score 128 x 4096^2 x 64: 668 against 682 us; with two or
    // five buffers, or a two-stage ring, it was slower).
    if (!pub.stream_k && !pl.rl && !pl.ck && kb == 1 && pl.epi == EPI_TMA &&
        find_tc_variant(pl.var.bn, pl.var.pair, EPI_TMA | EPI_SQ, 0, &h2v))
        pl.var = h2v;
    pub.stages = pl.var.stages;
    const int cl = pl.ck ? 2 : pair;  // CTAs per cluster
    pub.units = pub.stream_k ? pub.dp_tiles : tiles * pub.splits;
    pub.grid = pub.stream_k ? sk_groups * cl : std::min<int64_t>(pub.units, G) * cl;
    pub.workspace_bytes = pl.pack_a_bytes + pl.pack_b_bytes + pl.partial_bytes + pl.sk_w_bytes + pl.sk_ctr_bytes;
}

// Tile width of the small-problem kernel for this problem, or 0 when the persistent
// kernel takes it: every 64-wide block of K resident at once (at most 8 for 64-wide
// tiles, 6 for 128-wide ones), K-major operands that tensor copies address as they are,
// fp32 accumulation, and no option of the persistent kernel forced.
int small_plan_width(const Problem& pr, int sms) {
    const int64_t mode = g_opt_small.load();
    if (mode < 0) return 0;
    const int64_t kb = ceil_div(pr.K, 64);
    if (kb < 1 || pr.a_mn || pr.b_mn || pr.acc16 || pr.batch > 65535) return 0;
    if (!operand_tma_ok(pr.align & 1u, pr.lda, pr.sA, pr.batch) || !operand_tma_ok(pr.align & 2u, pr.ldb, pr.sB, pr.batch))
        return 0;
    if (g_opt_force_pack.load() || g_opt_skip_first_load.load()) return 0;
    const bool forced = g_opt_force_bn.load() || g_opt_force_pair.load() || g_opt_force_splits.load() ||
                        g_opt_force_swap.load() || g_opt_force_generic.load() || g_opt_stream_k.load() ||
                        g_opt_k_cluster.load() || g_opt_row_loader.load();
    if (forced) return 0;
    const int64_t tiles_m = ceil_div(pr.M, 128);
    const int64_t t128 = tiles_m * ceil_div(pr.N, 128) * pr.batch;
    // Automatic: 64-wide tiles when they fit one wave, where the persistent kernel's CTAs
    // would each run one tile and pay its set-up for it (back to back, GB300: 256^3 5.1
    // against 6.3 us, 1000^2 x 96 5.1 against 6.3, 300 x 264 x 256 with beta 6.1 against
    // 7.3, 512^3 6.4 against 8.3, 1024^2 x 512 6.3 against 8.3, 64 x 2048 x 512 6.3 against
    // 8.4).  With 128-wide tiles near a full wave it lost (1536^2 x 128: 7.1 against 6.4 us),
    // so larger problems stay on the persistent kernel.
    if (mode == 0 && 2 * t128 > sms) return 0;
    const int bn = (mode == 64 || mode == 128) ? static_cast<int>(mode) : (2 * t128 <= sms ? 64 : 128);
    if (kb > small_max_kb(bn) || ceil_div(pr.N, bn) > 65535) return 0;
    return bn;
}

// Tensor-core tile plan; pure host arithmetic, no CUDA calls.
void make_plan(const Problem& pr, int sms, Plan& pl, bool allow_small = true) {
    std::memset(&pl, 0, sizeof(pl));
    gemm_tn_plan_t& pub = pl.pub;
    pub.splits = 1;
    if (pr.M == 0 || pr.N == 0 || pr.batch == 0) {
        pub.kernel = 0;
        return;
    }
    if (pr.K == 0) {
        pub.kernel = 1;
        pub.units = pr.batch;
        return;
    }
    if (const int sbn = allow_small ? small_plan_width(pr, sms) : 0) {
        pl.small_bn = sbn;
        pub.kernel = 4;
        pub.tile_m = 128;
        pub.tile_n = sbn;
        pub.cta_pair = 1;
        pub.stages = static_cast<int32_t>(ceil_div(pr.K, 64));
        pub.units = ceil_div(pr.M, 128) * ceil_div(pr.N, sbn) * pr.batch;
        pub.grid = pub.units;
        return;
    }
    const bool force_pack = g_opt_force_pack.load() != 0;
    pub.pack_a = (force_pack || !operand_tma_ok(pr.align & 1u, pr.lda, pr.sA, pr.batch)) ? 1 : 0;
    pub.pack_b = (force_pack || !operand_tma_ok(pr.align & 2u, pr.ldb, pr.sB, pr.batch)) ? 1 : 0;
    const bool d_ok = operand_tma_ok(pr.align & 8u, pr.ldd, pr.sD, pr.batch);
    const bool c_ok = pr.beta == 0.0f || operand_tma_ok(pr.align & 4u, pr.ldc, pr.sC, pr.batch);

    // Small M: swap operands so that the long N side fills the 128 tensor-memory lanes
    // (K-major operands only: the swapped kernels have tiles narrower than an MN box).
    bool swap = pr.M <= 64 && pr.N >= 128 && pr.N >= 2 * pr.M;
    const int64_t fs = g_opt_force_swap.load();
    if (fs > 0 && pr.M <= 64) swap = true;
    if (fs < 0 || pr.a_mn || pr.b_mn || pr.acc16) swap = false;

    int bn, pair;
    const int64_t slots = std::max(sms, 1);
    if (swap) {
        bn = pr.M <= 16 ? 16 : pr.M <= 32 ? 32 : 64;
        pair = 1;
    } else {
        // 256x256 CTA-pair tiles are the most efficient shape; smaller tiles only
        // when short K or few tiles make the pair's fixed costs dominate.
        const int64_t t_pair = ceil_div(pr.M, 256) * ceil_div(pr.N, 256) * pr.batch;
        const int64_t t_256 = ceil_div(pr.M, 128) * ceil_div(pr.N, 256) * pr.batch;
        // 256x512 pair tiles halve the B rows loaded per MMA and measured faster only with
        // many full waves of long tiles (8192^3: 586-588 against 595-597 us); with fewer
        // waves the coarser quantisation loses (4096^3: 87.5 against 83-87 us, and their
        // 256 KB-per-CTA stream-K partials make the fix-up dearer than the idle wave: 98 us).
        const int64_t t_wide = ceil_div(pr.M, 256) * ceil_div(pr.N, 512) * pr.batch;
        const int64_t pairs = std::max<int64_t>(slots / 2, 1);
        const int64_t wide_tail = t_wide % pairs;
        const bool wide_ok = pr.K >= 8192 && t_wide >= 6 * pairs && (wide_tail == 0 || 10 * wide_tail >= 7 * pairs);
        // 256x432 pair tiles (MMAs of N = 256 and 176) where the waves of 512-column tiles
        // come out short: 6144 x 8192 x 8192 is exactly 6 waves of them (446 us against 475
        // for 256 x 256 tiles).  Where 512-column tiles qualify, the 432-column ones must
        // promise 5 % less MMA work on the critical path (waves x tile width): at the power
        // cap fewer idle SMs in a last wave raise the clock less than it seems, and 8192^3
        // measured the same either way (8 x 432 columns, 592-594 us, against 7 x 512,
        // 592-598), the 512-column tile moving fewer operand bytes per FLOP.  D = alpha A B^T
        // with K-major operands only.
        const int64_t t_432 = ceil_div(pr.M, 256) * ceil_div(pr.N, 432) * pr.batch;
        const int64_t tail_432 = t_432 % pairs;
        const bool k_major = !pr.a_mn && !pr.b_mn;
        if (pr.K >= 8192 && k_major && !pr.acc16 && pr.beta == 0.0f && t_432 >= 6 * pairs &&
            (tail_432 == 0 || 10 * tail_432 >= 7 * pairs) &&
            (!wide_ok || 20 * ceil_div(t_432, pairs) * 432 < 19 * ceil_div(t_wide, pairs) * 512)) {
            pair = 2;
            bn = 432;
        } else if (wide_ok) {
            pair = 2;
            bn = 512;
        } else if (pr.K >= 512 && 2 * t_pair >= slots) {
            pair = 2;
            bn = 256;
        } else if (t_256 >= slots || pr.N > 128 * 8) {
            // Under a wave of pair tiles, pairs and single CTAs with 128 x 256 tiles keep the
            // same SMs busy, and a pair loads 32 KB per SM and k-block where a single CTA
            // loads 48 KB for the same output: from 64 k-blocks on the pairs measured faster
            // (2048^2 x 8192 46.6 against 57.9 us, 1536^2 x 4096 28.8 against 33.0,
            // 1024 x 4096 x 4096 28.9 against 32.9), at 32 k-blocks even, at 16 slower.
            pair = pr.K >= 64 * 64 ? 2 : 1;
            bn = 256;
        } else {
            pair = 1;
            bn = 128;
        }
        const int64_t fbn = g_opt_force_bn.load(), fpair = g_opt_force_pair.load();
        if (fbn == 128 || fbn == 256 || fbn == 432 || fbn == 512) bn = static_cast<int>(fbn);
        if (fpair == 1 || fpair == 2) pair = static_cast<int>(fpair);
    }
    const int64_t rows_a = swap ? pr.N : pr.M;
    const int64_t rows_b = swap ? pr.M : pr.N;
    const int64_t kb = ceil_div(pr.K, 64);

    // Split-K with a separate reduction: when forced, and for K of 32 or more k-blocks on
    // tiles that would leave at least three quarters of the SMs idle.  There the K slices
    // fill the GPU (their fp32 partials leave by TMA) and the reduction kernel reads them
    // with every SM; the stream-K fix-up, one CTA per tile reading its contributors one
    // after another, measured slower (256 x 384 x 131072: 65 us stream-K, 75 with 8
    // slices, 472 data-parallel), and so did data-parallel tiles from 32 k-blocks on
    // (256 x 256 x 4096 22.1 against 14.0 us, 512 x 512 x 2048 15.9 against 14.5).  Other
    // shapes with too few tiles take the stream-K split decided in plan_stream_k.
    int splits = 1;
    const int64_t fsplit = g_opt_force_splits.load();
    const bool split_ok = !pr.a_mn && !pr.b_mn && !pr.acc16;
    if (fsplit >= 1 && split_ok) {
        pair = 1;
        splits = static_cast<int>(std::min<int64_t>(fsplit, kb));
        if (!swap) bn = 128;  // the partial-sum variant exists at 128 columns
    } else if (fsplit == 0 && split_ok && g_opt_stream_k.load() == 0 && kb >= 32) {
        if (!swap) {
            const int64_t t128 = ceil_div(pr.M, 128) * ceil_div(pr.N, 128) * pr.batch;
            // Up to half the SMs busy and 128-255 k-blocks: two slices measured faster too
            // (768 x 1280 x 8192 30.2 against 44.5 us, 1024^2 x 8192 30.7 against 33.9,
            // 640 x 1024 x 8192 28.7 against 30.2); from 256 k-blocks on it was mixed
            // (896 x 1024 x 16384 44.7 against 42.6, 1024^2 x 16384 45.1 against 46.6).
            const bool half = t128 * 2 <= slots && kb >= 128 && kb < 256;
            if (t128 * 4 <= slots || half) {
                pair = 1;
                bn = 128;
                splits = static_cast<int>(std::min<int64_t>({32, kb / 8, std::max<int64_t>(2, slots / t128)}));
            }
        } else {
            // swapped (small M): 128-row tiles along N.  With room for two or more slices per
            // tile in one wave and 64+ k-blocks, slices measured faster than stream-K or whole
            // tiles (48 x 1024 x 32768 27.9 against 40.8 us; 64 x 512 x 131072 39.4 against
            // 59.3; 64 x 8192 x 8192 33.7 against 40.3; 64 x 4096 x 4096 18.5 against 26.6;
            // 32 x 8192 x 4096 24.3 against 26.8), or tied (16 x 8192 x 8192 34.6 against 34.7).
            const int64_t tsw = ceil_div(pr.N, 128) * pr.batch;
            if (kb >= 64 && tsw * 2 <= slots)
                splits = static_cast<int>(std::min<int64_t>({32, kb / 8, slots / tsw}));
        }
    }
    // Two K halves of a swapped tile on the two CTAs of a cluster, the second half's partial
    // sum added by the first CTA through distributed shared memory: one launch and no scratch
    // where two K slices and a separate sum kernel would run (the 16 x 8192 x 8192 workload).
    const int64_t fck = g_opt_k_cluster.load();
    if (swap && fsplit == 0 && (fck > 0 || (fck == 0 && splits == 2)) && kb >= 2 &&
        find_tc_variant(bn, 1, EPI_SWAP | EPI_CK, 0, nullptr)) {
        splits = 1;
        pl.ck = 1;
    }

    // D rows TMA cannot address are written by the epilogue itself, each thread its row,
    // through the aligned 16-byte words that cover each row segment (EPI_VEC); C of any
    // alignment is read the same way (EPI_TMA_CG, EPI_VEC).  Against the predicated
    // epilogue, and against writing D by TMA to an aligned scratch copy moved into place
    // afterwards, this measured faster at every size: 4095 x 3073 x 2047 with ldd 3073
    // 59.5-60.4 against 64.4-64.9 us staged; 2048^2 x 1024 20.5 against 26.2; 512^3 12.3
    // against 16.4 predicated.
    const bool force_generic = g_opt_force_generic.load() != 0;
    const bool vec = !pr.acc16 && splits == 1 && !swap && !force_generic && !d_ok;
    int epi;
    if (pr.acc16) epi = (pr.beta == 0.0f && d_ok && !force_generic) ? EPI_TMA_A16 : EPI_GENERIC_A16;
    else if (splits > 1) epi = swap ? EPI_PARTIAL_SWAP : EPI_PARTIAL;
    else if (swap) epi = EPI_SWAP;
    else if (vec) epi = EPI_VEC;
    else if (d_ok && !force_generic) epi = pr.beta == 0.0f ? EPI_TMA : (c_ok ? EPI_TMA_C : EPI_TMA_CG);
    else epi = EPI_GENERIC;

    TcVariant v;
    // 432 columns: CTA pairs, D = alpha * acc by TMA stores; 512 columns: CTA pairs, TMA epilogues
    if (bn == 432 && (swap || pr.a_mn || pr.b_mn || !find_tc_variant(bn, pair, epi, 0, nullptr))) bn = 512;
    if (bn == 512 && !find_tc_variant(bn, pair, epi, 0, nullptr)) bn = 256;
    if (pl.ck) {
        find_tc_variant(bn, 1, EPI_SWAP | EPI_CK, 0, &v);
    } else if (!find_tc_variant(bn, pair, epi, 0, &v)) {
        // Fall back to the single-CTA variant of the same epilogue.
        pair = 1;
        if (!find_tc_variant(bn, pair, epi, 0, &v)) {
            bn = 128;
            find_tc_variant(bn, pair, epi, 0, &v);
        }
    }
    // Operands whose rows TMA cannot address are repacked to an aligned scratch copy first,
    // or, on request, read by the loader warps of a row-loader variant where one exists
    // (K-major, unswapped, whole tiles): no scratch, but slower -- the loader warps' loads,
    // one row per lane, cost about 2300 L1 wavefronts per k-block against the 512 cycles
    // its MMAs take (GB300: 4095 x 3073 x 2047 packed, 190.9 against 56.5 us repacked;
    // 4096^3 with lda = 4097, 591 against 81 us aligned).
    if (g_opt_row_loader.load() > 0 && (pub.pack_a || pub.pack_b) && !force_pack && !swap && !pr.a_mn && !pr.b_mn &&
        splits == 1) {
        TcVariant rv;
        if (find_tc_variant(v.bn, v.pair, epi | EPI_RL, 0, &rv)) {
            v = rv;
            pl.rl = 1;
            pl.rl_a = pub.pack_a;
            pl.rl_b = pub.pack_b;
            pub.pack_a = pub.pack_b = 0;
        }
    }
    pub.row_load = (pl.rl_a ? 1 : 0) | (pl.rl_b ? 2 : 0);
    pub.k_cluster = pl.ck;
    pl.var = v;
    pl.epi = epi;
    pl.rows_a = rows_a;
    pl.rows_b = rows_b;
    pl.tiles_m = ceil_div(rows_a, 128 * pair);
    pl.tiles_n = ceil_div(rows_b, bn);
    // 16 tile rows per rasterisation group (ncu, GB300: 4096^3 DRAM traffic 125.7 MB against
    // 151.9 MB with 8 rows, 85.4 against 86.1 us; 8192^3 with serpentine K order 831 MB
    // against 1019 MB with 8 rows and forward K order).
    pl.group_m = g_opt_group_m.load() > 0 ? static_cast<int>(g_opt_group_m.load()) : 16;

    pub.kernel = splits > 1 ? 3 : 2;
    pub.tile_m = 128 * pair;
    pub.tile_n = bn;
    pub.cta_pair = pair;
    pub.swap_ab = swap ? 1 : 0;
    pub.splits = splits;
    pub.stages = v.stages;
    pub.epi_tma = (epi_base(epi) == EPI_TMA || epi == EPI_TMA_C || epi == EPI_TMA_CG) ? 1 : 0;

    pl.ldo_a = round_up(a_len(pr), 8);
    pl.ldo_b = round_up(b_len(pr), 8);
    const int64_t nba = (pr.batch > 1 && pr.sA != 0) ? pr.batch : 1;
    const int64_t nbb = (pr.batch > 1 && pr.sB != 0) ? pr.batch : 1;
    pl.pack_a_bytes = pub.pack_a ? round_up(nba * a_rows(pr) * pl.ldo_a * 2, 256) : 0;
    pl.pack_b_bytes = pub.pack_b ? round_up(nbb * b_rows(pr) * pl.ldo_b * 2, 256) : 0;
    pl.partial_bytes = splits > 1 ? round_up(pr.batch * splits * pr.M * pr.N * 4, 256) : 0;
    plan_stream_k(pr, pl, slots / (pl.ck ? 2 : pair));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ranges_overlap(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

int64_t extent_bytes(int64_t rows, int64_t cols, int64_t ld, int64_t stride, int64_t batch) {
    return 2 * ((batch - 1) * stride + (rows - 1) * ld + cols);
}

// Byte range of a matrix for the checked build's device-side bounds checks.
Extent extent_of(const void* base, int64_t bytes) {
    const uint64_t lo = static_cast<uint64_t>(reinterpret_cast<uintptr_t>(base));
    return Extent{lo, lo + static_cast<uint64_t>(bytes > 0 ? bytes : 0)};
}

gemm_status_t run(const void* A, const void* B, const void* C, void* D, const Problem& pr, float alpha,
                  cudaStream_t stream) {
    gemm_status_t st = validate(pr);
    if (st != GEMM_OK) return st;
    if (pr.M == 0 || pr.N == 0 || pr.batch == 0) return GEMM_OK;
    if (!D) return GEMM_ERR_INVALID_VALUE;
    if (pr.K > 0 && (!A || !B)) return GEMM_ERR_INVALID_VALUE;
    if (pr.beta != 0.0f && !C) return GEMM_ERR_INVALID_VALUE;
    auto odd = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) != 0; };
    if (odd(D) || (pr.K > 0 && (odd(A) || odd(B))) || (pr.beta != 0.0f && odd(C))) return GEMM_ERR_MISALIGNED;

    // D must not overlap any input, except C exactly.
    const int64_t d_bytes = extent_bytes(pr.M, pr.N, pr.ldd, pr.sD, pr.batch);
    if (pr.K > 0) {
        if (ranges_overlap(D, d_bytes, A, extent_bytes(a_rows(pr), a_len(pr), pr.lda, pr.sA, pr.batch)) ||
            ranges_overlap(D, d_bytes, B, extent_bytes(b_rows(pr), b_len(pr), pr.ldb, pr.sB, pr.batch)))
            return GEMM_ERR_INVALID_VALUE;
    }
    if (pr.beta != 0.0f) {
        if (C == D) {
            if (pr.ldc != pr.ldd || (pr.batch > 1 && pr.sC != pr.sD)) return GEMM_ERR_INVALID_VALUE;
        } else if (ranges_overlap(D, d_bytes, C, extent_bytes(pr.M, pr.N, pr.ldc, pr.sC, pr.batch))) {
            return GEMM_ERR_INVALID_VALUE;
        }
    }

    DeviceState* dev = nullptr;
    if ((st = device_state(&dev)) != GEMM_OK) return st;

    cudaError_t e;
    if (pr.K == 0) {
        ReduceChecks chk = {};
        chk.c = pr.beta != 0.0f ? extent_of(C, extent_bytes(pr.M, pr.N, pr.ldc, pr.sC, pr.batch)) : Extent{};
        chk.d = extent_of(D, d_bytes - g_opt_check_trim_d.load());
        chk.err = dev->err;
        e = launch_scale(pr.M, pr.N, pr.batch, pr.beta, C, pr.ldc, pr.sC, D, pr.ldd, pr.sD, dev->sms, stream, chk);
        return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
    }

    Problem p = pr;
    p.align = (aligned16(A) ? 1u : 0u) | (aligned16(B) ? 2u : 0u) | (aligned16(C) ? 4u : 0u) |
              (aligned16(D) ? 8u : 0u);
    Plan pl;
    make_plan(p, dev->sms, pl);

    if (pl.small_bn > 0) {
        // Small-problem kernel: operands read in place by tensor copies (boxes of 64 K x 128
        // rows of A and 64 K x tile_n rows of B); should the driver refuse a map, the
        // persistent kernel's plan takes over.
        const bool a_b = p.batch > 1 && p.sA != 0, b_b = p.batch > 1 && p.sB != 0;
        CUtensorMap sA_map, sB_map;
        if (encode_map(&sA_map, A, p.K, p.M, p.batch, p.lda, p.sA, a_b, 64, 128) &&
            encode_map(&sB_map, B, p.K, p.N, p.batch, p.ldb, p.sB, b_b, 64, static_cast<uint32_t>(pl.small_bn))) {
            SmallParams sp;
            std::memset(&sp, 0, sizeof(sp));
            sp.M = static_cast<int32_t>(p.M);
            sp.N = static_cast<int32_t>(p.N);
            sp.kb = static_cast<int32_t>(ceil_div(p.K, 64));
            sp.zA = a_b ? 1 : 0;
            sp.zB = b_b ? 1 : 0;
            sp.alpha = alpha;
            sp.beta = p.beta;
            sp.C = C;
            sp.ldc = p.ldc;
            sp.strideC = p.batch > 1 ? p.sC : 0;
            sp.D = D;
            sp.ldd = p.ldd;
            sp.strideD = p.batch > 1 ? p.sD : 0;
            sp.err = dev->err;
            sp.timeout_ns = static_cast<uint64_t>(g_opt_timeout_ns.load());
            sp.ext_c = p.beta != 0.0f
                           ? extent_of(C, extent_bytes(p.M, p.N, p.ldc, p.sC, (p.batch > 1 && p.sC != 0) ? p.batch : 1))
                           : Extent{};
            sp.ext_d = extent_of(D, d_bytes - g_opt_check_trim_d.load());
            e = launch_small_gemm(sA_map, sB_map, sp, pl.small_bn, ceil_div(p.M, 128), ceil_div(p.N, pl.small_bn),
                                  p.batch, stream);
            return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
        }
        make_plan(p, dev->sms, pl, false);
    }

    // Tensor maps first: an operand whose map the driver rejects is repacked instead.
    const bool swap = pl.pub.swap_ab != 0;
    // B rows per box: one box per MMA of N <= 256 columns, split between a CTA pair
    const uint32_t box_rows_b = static_cast<uint32_t>(std::min(pl.var.bn, 256) / pl.var.pair);
    CUtensorMap mapA_op, mapB_op, mapC, mapD;
    std::memset(&mapC, 0, sizeof(mapC));
    std::memset(&mapD, 0, sizeof(mapD));
    // Problem operand A is the MMA's B operand when swapped, else its A operand.  A
    // K-major operand is fetched in boxes of 64 K x rows, an MN-major one in boxes of
    // 64 (M or N) x 64 K.
    const uint32_t boxA = p.a_mn ? 64u : (swap ? box_rows_b : 128u);
    const uint32_t boxB = p.b_mn ? 64u : (swap ? 128u : box_rows_b);
    CUtensorMap mapPA, mapPB;
    std::memset(&mapPA, 0, sizeof(mapPA));  // operands read by the row loader need no map
    std::memset(&mapPB, 0, sizeof(mapPB));
    if (!pl.pub.pack_a && !pl.rl_a && !encode_map(&mapPA, A, a_len(p), a_rows(p), p.batch, p.lda, p.sA, p.batch > 1 && p.sA != 0,
                                      64, boxA))
        pl.pub.pack_a = 1,
        pl.pack_a_bytes = round_up(((p.batch > 1 && p.sA != 0) ? p.batch : 1) * a_rows(p) * pl.ldo_a * 2, 256);
    if (!pl.pub.pack_b && !pl.rl_b && !encode_map(&mapPB, B, b_len(p), b_rows(p), p.batch, p.ldb, p.sB, p.batch > 1 && p.sB != 0,
                                      64, boxB))
        pl.pub.pack_b = 1,
        pl.pack_b_bytes = round_up(((p.batch > 1 && p.sB != 0) ? p.batch : 1) * b_rows(p) * pl.ldo_b * 2, 256);
    if ((epi_base(pl.epi) == EPI_TMA || pl.epi == EPI_TMA_C || pl.epi == EPI_TMA_CG) &&
        (!encode_map(&mapD, D, p.N, p.M, p.batch, p.ldd, p.sD, p.batch > 1, 64, 32) ||
         (pl.epi == EPI_TMA_C &&
          !encode_map(&mapC, C, p.N, p.M, p.batch, p.ldc, p.sC, p.batch > 1 && p.sC != 0, 64, 32)))) {
        TcVariant v;
        const int generic = epi_acc16(pl.epi) ? EPI_GENERIC_A16 : EPI_GENERIC;
        // (512-column tiles exist with TMA epilogues only: 256 columns, same B boxes)
        if (find_tc_variant(pl.var.bn, pl.var.pair, generic, 0, &v) ||
            find_tc_variant(std::min(pl.var.bn, 256), pl.var.pair, generic, 0, &v)) {
            if (pl.rl) {  // no row-loader variant with this epilogue: repack those operands
                pl.pub.pack_a |= pl.rl_a;
                pl.pub.pack_b |= pl.rl_b;
                pl.pack_a_bytes = pl.pub.pack_a
                    ? round_up(((p.batch > 1 && p.sA != 0) ? p.batch : 1) * a_rows(p) * pl.ldo_a * 2, 256) : 0;
                pl.pack_b_bytes = pl.pub.pack_b
                    ? round_up(((p.batch > 1 && p.sB != 0) ? p.batch : 1) * b_rows(p) * pl.ldo_b * 2, 256) : 0;
                pl.rl = pl.rl_a = pl.rl_b = 0;
                pl.pub.row_load = 0;
            }
            pl.var = v;
            pl.epi = generic;
            pl.pub.epi_tma = 0;
            pl.pub.stages = v.stages;
            pl.pub.tile_n = v.bn;
            pl.tiles_n = ceil_div(pl.rows_b, v.bn);
        } else {
            return GEMM_ERR_UNSUPPORTED;
        }
    }

    int64_t cap = dev->capacity[pl.var.index];
    if (cap == 0) {
        cap = tc_variant_capacity(pl.var, dev->sms);
        if (cap <= 0) cap = dev->sms;
        dev->capacity[pl.var.index] = cap;
    }
    plan_stream_k(p, pl, cap / (pl.ck ? 2 : pl.var.pair));

    const int64_t ws_bytes = pl.pack_a_bytes + pl.pack_b_bytes + pl.partial_bytes + pl.sk_w_bytes + pl.sk_ctr_bytes;
    uint8_t* ws = nullptr;
    if (ws_bytes > 0) {
        e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws), static_cast<size_t>(ws_bytes), dev->pool, stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_WORKSPACE;
        }
    }
    auto release = [&]() {
        if (ws) cudaFreeAsync(ws, stream);
    };

    const bool a_batched = p.batch > 1 && p.sA != 0;
    const bool b_batched = p.batch > 1 && p.sB != 0;
    RepackArgs jobs[2];
    int njobs = 0;
    if (pl.pub.pack_a) {
        void* dst = ws;
        jobs[njobs++] = {A, p.lda, p.sA, dst, pl.ldo_a, a_rows(p), a_len(p), a_batched ? p.batch : 1,
                         extent_of(A, extent_bytes(a_rows(p), a_len(p), p.lda, p.sA, a_batched ? p.batch : 1)),
                         extent_of(dst, pl.pack_a_bytes)};
        if (!encode_map(&mapPA, dst, a_len(p), a_rows(p), p.batch, pl.ldo_a, a_rows(p) * pl.ldo_a, a_batched, 64,
                        boxA)) {
            release();
            return GEMM_ERR_UNSUPPORTED;
        }
    }
    if (pl.pub.pack_b) {
        void* dst = ws + pl.pack_a_bytes;
        jobs[njobs++] = {B, p.ldb, p.sB, dst, pl.ldo_b, b_rows(p), b_len(p), b_batched ? p.batch : 1,
                         extent_of(B, extent_bytes(b_rows(p), b_len(p), p.ldb, p.sB, b_batched ? p.batch : 1)),
                         extent_of(dst, pl.pack_b_bytes)};
        if (!encode_map(&mapPB, dst, b_len(p), b_rows(p), p.batch, pl.ldo_b, b_rows(p) * pl.ldo_b, b_batched, 64,
                        boxB)) {
            release();
            return GEMM_ERR_UNSUPPORTED;
        }
    }
    if (njobs > 0) {
        e = launch_repack(jobs, njobs, dev->sms, stream, dev->err);
        if (e != cudaSuccess) { release(); return cuda_fail(e); }
    }
    mapA_op = swap ? mapPB : mapPA;
    mapB_op = swap ? mapPA : mapPB;
    if (epi_base(pl.epi) != EPI_TMA && pl.epi != EPI_TMA_C && pl.epi != EPI_TMA_CG) mapD = mapA_op;  // unused by the kernel; any valid map
    if (pl.epi != EPI_TMA_C) mapC = mapD;

    KParams kp;
    std::memset(&kp, 0, sizeof(kp));
    kp.rows_a = static_cast<int32_t>(pl.rows_a);
    kp.rows_b = static_cast<int32_t>(pl.rows_b);
    kp.K = static_cast<int32_t>(p.K);
    kp.batch = static_cast<int32_t>(p.batch);
    kp.tiles_m = static_cast<int32_t>(pl.tiles_m);
    kp.tiles_n = static_cast<int32_t>(pl.tiles_n);
    kp.splits = pl.pub.splits;
    kp.kb_total = static_cast<int32_t>(ceil_div(p.K, 64));
    kp.group_m = pl.group_m;
    {
        // Serpentine K order where the operands are too large to stay in L2 between two
        // waves of data-parallel tiles.  An LRU model of the tile order reproduces the
        // measured DRAM reads of 8192^3 (881 / 822 / 847 MB for groups of 8 / 12 / 16 tile
        // rows) with about 50 MB of effective L2, and predicted 708 MB with serpentine order
        // and 16-row groups; ncu measured 712 MB.
        const int64_t mode = g_opt_serpentine.load();
        const int64_t groups = std::max<int64_t>(pl.pub.grid / pl.var.pair, 1);
        const int64_t op_bytes = 2 * (a_rows(p) * a_len(p) + b_rows(p) * b_len(p)) *
                                 ((p.batch > 1 && (p.sA != 0 || p.sB != 0)) ? p.batch : 1);
        kp.serp = (mode > 0 || (mode == 0 && pl.pub.dp_tiles >= 2 * groups && op_bytes >= (int64_t(128) << 20))) ? 1 : 0;
    }
    kp.zA = swap ? (b_batched ? 1 : 0) : (a_batched ? 1 : 0);
    kp.zB = swap ? (a_batched ? 1 : 0) : (b_batched ? 1 : 0);
    kp.zC = (p.batch > 1 && p.sC != 0) ? 1 : 0;
    kp.zD = p.batch > 1 ? 1 : 0;
    kp.a_mn = p.a_mn;  // operands are never swapped when one is MN-major
    kp.b_mn = p.b_mn;
    kp.num_units = pl.pub.units;
    kp.M = static_cast<int32_t>(p.M);
    kp.N = static_cast<int32_t>(p.N);
    kp.alpha = alpha;
    kp.beta = p.beta;
    kp.D = D;
    kp.ldd = p.ldd;
    kp.strideD = p.sD;
    kp.C = C;
    kp.ldc = p.ldc;
    kp.strideC = p.sC;
    kp.W = pl.pub.splits > 1 ? reinterpret_cast<float*>(ws + pl.pack_a_bytes + pl.pack_b_bytes) : nullptr;
    kp.err = dev->err;
    kp.timeout_ns = static_cast<uint64_t>(g_opt_timeout_ns.load());
    kp.debug_skip_first_load = g_opt_skip_first_load.load() != 0 ? 1 : 0;
    kp.ext_a = extent_of(A, extent_bytes(a_rows(p), a_len(p), p.lda, p.sA, a_batched ? p.batch : 1));
    kp.ext_b = extent_of(B, extent_bytes(b_rows(p), b_len(p), p.ldb, p.sB, b_batched ? p.batch : 1));
    kp.ext_c = p.beta != 0.0f ? extent_of(C, extent_bytes(p.M, p.N, p.ldc, p.sC, (p.batch > 1 && p.sC != 0) ? p.batch : 1))
                              : Extent{};
    kp.ext_d = extent_of(D, d_bytes - g_opt_check_trim_d.load());
    kp.ext_w = extent_of(kp.W, pl.partial_bytes);
    kp.pdl = njobs > 0 ? 1 : 0;  // directly behind the repack launch
    if (pl.rl) {
        // row loader: the MMA's operands are the problem's A and B (never swapped)
        kp.rl_on[0] = pl.rl_a;
        kp.rl_on[1] = pl.rl_b;
        kp.rl_ptr[0] = A;
        kp.rl_ptr[1] = B;
        kp.rl_ld[0] = p.lda;
        kp.rl_ld[1] = p.ldb;
        kp.rl_stride[0] = p.batch > 1 ? p.sA : 0;
        kp.rl_stride[1] = p.batch > 1 ? p.sB : 0;
        const int64_t a_box = 128 * 64 * 2, b_box = static_cast<int64_t>(pl.var.bn / pl.var.pair) * 64 * 2;
        kp.tma_tx = static_cast<uint32_t>(((pl.rl_a ? 0 : a_box) + (pl.rl_b ? 0 : b_box)) * pl.var.pair);
    }
    if (pl.epi == EPI_PARTIAL && encode_partials_map(&mapD, kp.W, p.M, p.N, p.batch * pl.pub.splits)) kp.w_tma = 1;

    if (pl.sk_iters > 0) {
        uint8_t* sk_base = ws + pl.pack_a_bytes + pl.pack_b_bytes + pl.partial_bytes;
        kp.sk_iters = pl.sk_iters;
        kp.sk_maxc = pl.pub.sk_maxc;
        kp.sk_W = reinterpret_cast<float*>(sk_base);
        kp.sk_counters = reinterpret_cast<unsigned long long*>(sk_base + pl.sk_w_bytes);
        kp.sk_epoch = next_sk_epoch();
    }
    int64_t grid = 0;
    e = launch_tc_variant(pl.var, mapA_op, mapB_op, mapC, mapD, kp, pl.pub.grid, stream, &grid);
    if (e != cudaSuccess) { release(); return cuda_fail(e); }
    if (pl.pub.splits > 1) {
        const ReduceChecks chk = {kp.ext_w, kp.ext_c, kp.ext_d, dev->err};
        e = launch_splitk_reduce(kp.W, pl.pub.splits, p.M, p.N, p.batch, alpha, p.beta, C, p.ldc, p.sC, D, p.ldd,
                                 p.sD, dev->sms, stream, chk);
        if (e != cudaSuccess) { release(); return cuda_fail(e); }
    }
    release();
    return GEMM_OK;
}

// ------------------------------------------------------------------ host-buffer GEMM

// D = alpha A B^T + beta C with every matrix in host memory.  B (N x K) goes to the
// device first; A, C and D travel in blocks of rows, so that block j's GEMM runs while
// block j+1's A and C come in and block j-1's D goes out.  Copies use two library
// streams joined to the caller's stream by events; device buffers come from the pool.
gemm_status_t run_host(const void* A, int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc, void* D,
                       int64_t ldd, int64_t M, int64_t N, int64_t K, float alpha, float beta, cudaStream_t stream) {
    Problem pr = {M, N, K, 1, lda, ldb, ldc, ldd, 0, 0, 0, 0, beta, 0};
    gemm_status_t st = validate(pr);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!D || (K > 0 && (!A || !B)) || (beta != 0.0f && !C)) return GEMM_ERR_INVALID_VALUE;
    auto odd = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 1u) != 0; };
    if (odd(D) || (K > 0 && (odd(A) || odd(B))) || (beta != 0.0f && odd(C))) return GEMM_ERR_MISALIGNED;
    // same aliasing rules as the device call: D overlaps no input, except C exactly
    const int64_t d_ext = extent_bytes(M, N, ldd, 0, 1);
    if (K > 0 && (ranges_overlap(D, d_ext, A, extent_bytes(M, K, lda, 0, 1)) ||
                  ranges_overlap(D, d_ext, B, extent_bytes(N, K, ldb, 0, 1))))
        return GEMM_ERR_INVALID_VALUE;
    if (beta != 0.0f && (C == D ? ldc != ldd : ranges_overlap(D, d_ext, C, extent_bytes(M, N, ldc, 0, 1))))
        return GEMM_ERR_INVALID_VALUE;
    DeviceState* dev = nullptr;
    if ((st = device_state(&dev)) != GEMM_OK) return st;
    cudaError_t e;
    {
        std::lock_guard<std::mutex> lock(g_dev_mu);
        if (!dev->copy_in && (e = cudaStreamCreateWithFlags(&dev->copy_in, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e);
        if (!dev->copy_out && (e = cudaStreamCreateWithFlags(&dev->copy_out, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e);
    }
    const bool use_c = beta != 0.0f;
    const int64_t a_bytes = K > 0 ? 2 * ((M - 1) * lda + K) : 0;
    const int64_t b_bytes = K > 0 ? 2 * ((N - 1) * ldb + K) : 0;
    const int64_t c_bytes = use_c ? 2 * ((M - 1) * ldc + N) : 0;
    const int64_t d_bytes = 2 * ((M - 1) * ldd + N);
    const int64_t a_off = 0, b_off = round_up(a_bytes, 256), c_off = b_off + round_up(b_bytes, 256),
                  d_off = c_off + round_up(c_bytes, 256), total = d_off + round_up(d_bytes, 256);
    uint8_t* buf = nullptr;
    if ((e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&buf), static_cast<size_t>(total), dev->pool, stream)) !=
        cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_WORKSPACE;
    }
    // Row blocks: about four, 512 to 1024 rows each (multiples of the 256-row tile).  On
    // 4096^3, 512- or 256-row blocks measured slower (more, smaller GEMMs in the chain);
    // on 8192^3 eight 1024-row blocks beat four 2048-row ones (1.65 against 1.74 ms).
    const int64_t rows_blk = std::min<int64_t>(1024, std::max<int64_t>(512, round_up(ceil_div(M, 4), 256)));
    const int64_t nblk = ceil_div(M, rows_blk);
    std::vector<cudaEvent_t> evs;
    auto new_event = [&](cudaEvent_t* ev) {
        cudaError_t r = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (r == cudaSuccess) evs.push_back(*ev);
        return r;
    };
    auto finish = [&](gemm_status_t status) {
        for (cudaEvent_t ev : evs) cudaEventDestroy(ev);  // released once pending work completes
        return status;
    };
    auto fail = [&](cudaError_t r) {
        // join the copy streams before the buffer goes back to the pool
        cudaEvent_t ev_in = nullptr, ev_out = nullptr;
        if (new_event(&ev_in) == cudaSuccess && cudaEventRecord(ev_in, dev->copy_in) == cudaSuccess)
            cudaStreamWaitEvent(stream, ev_in, 0);
        if (new_event(&ev_out) == cudaSuccess && cudaEventRecord(ev_out, dev->copy_out) == cudaSuccess)
            cudaStreamWaitEvent(stream, ev_out, 0);
        cudaFreeAsync(buf, stream);
        return finish(cuda_fail(r));
    };
    cudaEvent_t ev_start;
    if ((e = new_event(&ev_start)) != cudaSuccess || (e = cudaEventRecord(ev_start, stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(dev->copy_in, ev_start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(dev->copy_out, ev_start, 0)) != cudaSuccess)
        return fail(e);
    uint8_t* dA = buf + a_off;
    uint8_t* dB = buf + b_off;
    uint8_t* dC = buf + c_off;
    uint8_t* dD = buf + d_off;
    // rows x width halves of a row-major matrix with leading dimension ld: only the
    // elements travel, never the padding between rows
    auto copy_rows = [&](void* dst, const void* src, int64_t ld, int64_t width, int64_t rows, cudaMemcpyKind kind,
                         cudaStream_t s_) {
        return cudaMemcpy2DAsync(dst, static_cast<size_t>(2 * ld), src, static_cast<size_t>(2 * ld),
                                 static_cast<size_t>(2 * width), static_cast<size_t>(rows), kind, s_);
    };
    if (K > 0 && (e = copy_rows(dB, B, ldb, K, N, cudaMemcpyHostToDevice, dev->copy_in)) != cudaSuccess) return fail(e);
    for (int64_t j = 0; j < nblk; ++j) {
        const int64_t r0 = j * rows_blk, rows = std::min(rows_blk, M - r0);
        if (K > 0 && (e = copy_rows(dA + 2 * r0 * lda, static_cast<const uint8_t*>(A) + 2 * r0 * lda, lda, K, rows,
                                    cudaMemcpyHostToDevice, dev->copy_in)) != cudaSuccess)
            return fail(e);
        if (use_c && (e = copy_rows(dC + 2 * r0 * ldc, static_cast<const uint8_t*>(C) + 2 * r0 * ldc, ldc, N, rows,
                                    cudaMemcpyHostToDevice, dev->copy_in)) != cudaSuccess)
            return fail(e);
        cudaEvent_t ev_in, ev_done;
        if ((e = new_event(&ev_in)) != cudaSuccess || (e = cudaEventRecord(ev_in, dev->copy_in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(stream, ev_in, 0)) != cudaSuccess)
            return fail(e);
        Problem pj = {rows, N, K, 1, lda, ldb, ldc, ldd, 0, 0, 0, 0, beta, 0};
        st = run(dA + 2 * r0 * lda, dB, use_c ? dC + 2 * r0 * ldc : nullptr, dD + 2 * r0 * ldd, pj, alpha, stream);
        if (st != GEMM_OK) {
            fail(cudaSuccess);
            return st;
        }
        if ((e = new_event(&ev_done)) != cudaSuccess || (e = cudaEventRecord(ev_done, stream)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(dev->copy_out, ev_done, 0)) != cudaSuccess)
            return fail(e);
        if ((e = copy_rows(static_cast<uint8_t*>(D) + 2 * r0 * ldd, dD + 2 * r0 * ldd, ldd, N, rows,
                           cudaMemcpyDeviceToHost, dev->copy_out)) != cudaSuccess)
            return fail(e);
    }
    cudaEvent_t ev_end;
    if ((e = new_event(&ev_end)) != cudaSuccess || (e = cudaEventRecord(ev_end, dev->copy_out)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, ev_end, 0)) != cudaSuccess)
        return fail(e);
    if ((e = cudaFreeAsync(buf, stream)) != cudaSuccess) return finish(cuda_fail(e));
    return finish(GEMM_OK);
}

// Fused score + softmax statistics: validation, optional repack of operands TMA
// cannot fetch as they are, tensor maps, launch.
gemm_status_t run_softmax(const void* Q, int64_t ldq, int64_t strideQ, const void* K, int64_t ldk, int64_t strideK,
                          float* row_max, float* row_sum, int64_t M, int64_t N, int64_t d, int64_t batch, float alpha,
                          cudaStream_t stream) {
    if (M < 0 || N < 0 || d < 0 || batch < 0) return GEMM_ERR_INVALID_VALUE;
    const int64_t lim = int64_t(1) << 31;
    if (M >= lim || N >= lim || batch >= lim) return GEMM_ERR_UNSUPPORTED;
    if (d > 256) return GEMM_ERR_UNSUPPORTED;
    if (M == 0 || batch == 0) return GEMM_OK;
    if (!row_max || !row_sum) return GEMM_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(row_max) & 3u) || (reinterpret_cast<uintptr_t>(row_sum) & 3u))
        return GEMM_ERR_MISALIGNED;
    const int64_t rows = batch * M;
    if (ranges_overlap(row_max, 4 * rows, row_sum, 4 * rows)) return GEMM_ERR_INVALID_VALUE;
    const bool live = N > 0 && d > 0;  // otherwise the statistics are constants
    if (live) {
        if (!Q || !K || ldq < d || ldk < d) return GEMM_ERR_INVALID_VALUE;
        if (batch > 1 && (strideQ < 0 || strideK < 0)) return GEMM_ERR_INVALID_VALUE;
        if ((reinterpret_cast<uintptr_t>(Q) & 1u) || (reinterpret_cast<uintptr_t>(K) & 1u)) return GEMM_ERR_MISALIGNED;
        const int64_t q_bytes = extent_bytes(M, d, ldq, strideQ, batch);
        const int64_t k_bytes = extent_bytes(N, d, ldk, strideK, batch);
        if (ranges_overlap(row_max, 4 * rows, Q, q_bytes) || ranges_overlap(row_sum, 4 * rows, Q, q_bytes) ||
            ranges_overlap(row_max, 4 * rows, K, k_bytes) || ranges_overlap(row_sum, 4 * rows, K, k_bytes))
            return GEMM_ERR_INVALID_VALUE;
    }

    DeviceState* dev = nullptr;
    gemm_status_t st = device_state(&dev);
    if (st != GEMM_OK) return st;
    cudaError_t e;
    if (!live) {
        // N == 0: empty maximum and sum.  d == 0: every score is 0, so m = 0 and l = N.
        const float mv = N == 0 ? -std::numeric_limits<float>::infinity() : 0.0f;
        const float lv = static_cast<float>(N);
        e = launch_fill_stats(row_max, row_sum, rows, mv, lv, dev->sms, stream);
        return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
    }

    const bool q_batched = batch > 1 && strideQ != 0;
    const bool k_batched = batch > 1 && strideK != 0;
    const int kq = d <= 64 ? 1 : d <= 128 ? 2 : 4;
    CUtensorMap mapQ, mapK;
    bool pack_q = !operand_tma_ok(aligned16(Q), ldq, strideQ, q_batched ? batch : 1) ||
                  !encode_map(&mapQ, Q, d, M, batch, ldq, strideQ, q_batched, 64, kSoftmaxTileM);
    const uint32_t key_box = static_cast<uint32_t>(softmax_tile_n());
    bool pack_k = !operand_tma_ok(aligned16(K), ldk, strideK, k_batched ? batch : 1) ||
                  !encode_map(&mapK, K, d, N, batch, ldk, strideK, k_batched, 64, key_box);
    const int64_t ldo = round_up(d, 8);
    const int64_t q_pack_bytes = pack_q ? round_up((q_batched ? batch : 1) * M * ldo * 2, 256) : 0;
    const int64_t k_pack_bytes = pack_k ? round_up((k_batched ? batch : 1) * N * ldo * 2, 256) : 0;
    uint8_t* ws = nullptr;
    if (q_pack_bytes + k_pack_bytes > 0) {
        e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws), static_cast<size_t>(q_pack_bytes + k_pack_bytes),
                                    dev->pool, stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_WORKSPACE;
        }
    }
    auto release = [&]() {
        if (ws) cudaFreeAsync(ws, stream);
    };
    RepackArgs jobs[2];
    int njobs = 0;
    if (pack_q) {
        jobs[njobs++] = {Q, ldq, strideQ, ws, ldo, M, d, q_batched ? batch : 1,
                         extent_of(Q, extent_bytes(M, d, ldq, strideQ, q_batched ? batch : 1)),
                         extent_of(ws, q_pack_bytes)};
        if (!encode_map(&mapQ, ws, d, M, batch, ldo, M * ldo, q_batched, 64, kSoftmaxTileM)) {
            release();
            return GEMM_ERR_UNSUPPORTED;
        }
    }
    if (pack_k) {
        jobs[njobs++] = {K, ldk, strideK, ws + q_pack_bytes, ldo, N, d, k_batched ? batch : 1,
                         extent_of(K, extent_bytes(N, d, ldk, strideK, k_batched ? batch : 1)),
                         extent_of(ws + q_pack_bytes, k_pack_bytes)};
        if (!encode_map(&mapK, ws + q_pack_bytes, d, N, batch, ldo, N * ldo, k_batched, 64, key_box)) {
            release();
            return GEMM_ERR_UNSUPPORTED;
        }
    }
    if (njobs > 0) {
        e = launch_repack(jobs, njobs, dev->sms, stream, dev->err);
        if (e != cudaSuccess) { release(); return cuda_fail(e); }
    }

    SoftmaxParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.M = static_cast<int32_t>(M);
    sp.N = static_cast<int32_t>(N);
    sp.mblocks = static_cast<int32_t>(ceil_div(M, kSoftmaxTileM));
    sp.ntiles = static_cast<int32_t>(ceil_div(N, softmax_tile_n()));
    sp.num_units = batch * sp.mblocks;
    sp.alpha = alpha;
    sp.sc = static_cast<float>(static_cast<double>(alpha) * 1.4426950408889634074);  // alpha * log2(e)
    sp.row_max = row_max;
    sp.row_sum = row_sum;
    sp.err = dev->err;
    sp.timeout_ns = static_cast<uint64_t>(g_opt_timeout_ns.load());
    sp.zq = q_batched ? 1 : 0;
    sp.zk = k_batched ? 1 : 0;
    e = launch_score_softmax(mapQ, mapK, sp, kq, dev->sms, stream);
    release();
    return e == cudaSuccess ? GEMM_OK : cuda_fail(e);
}

}  // namespace
}  // namespace gtn

using namespace gtn;

extern "C" {

gemm_status_t gemm_tn_f16(const void* A, int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc,
                          void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                          gemm_stream_t stream) {
    Problem p = {M, N, K, 1, lda, ldb, ldc, ldd, 0, 0, 0, 0, beta, 0};
    return run(A, B, C, D, p, alpha, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_tn_f16_batched(const void* A, int64_t lda, int64_t strideA, const void* B, int64_t ldb,
                                  int64_t strideB, const void* C, int64_t ldc, int64_t strideC, void* D, int64_t ldd,
                                  int64_t strideD, int64_t M, int64_t N, int64_t K, int64_t batch, float alpha,
                                  float beta, gemm_stream_t stream) {
    Problem p = {M, N, K, batch, lda, ldb, ldc, ldd, strideA, strideB, strideC, strideD, beta, 0};
    return run(A, B, C, D, p, alpha, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f16(int32_t a_major, int32_t b_major, const void* A, int64_t lda, int64_t strideA, const void* B,
                       int64_t ldb, int64_t strideB, const void* C, int64_t ldc, int64_t strideC, void* D, int64_t ldd,
                       int64_t strideD, int64_t M, int64_t N, int64_t K, int64_t batch, float alpha, float beta,
                       gemm_stream_t stream) {
    if ((a_major != GEMM_K_MAJOR && a_major != GEMM_MN_MAJOR) || (b_major != GEMM_K_MAJOR && b_major != GEMM_MN_MAJOR))
        return GEMM_ERR_INVALID_VALUE;
    Problem p = {M, N, K, batch, lda, ldb, ldc, ldd, strideA, strideB, strideC, strideD, beta, 0};
    p.a_mn = a_major == GEMM_MN_MAJOR ? 1 : 0;
    p.b_mn = b_major == GEMM_MN_MAJOR ? 1 : 0;
    return run(A, B, C, D, p, alpha, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f16_acc16(int32_t a_major, int32_t b_major, const void* A, int64_t lda, int64_t strideA,
                             const void* B, int64_t ldb, int64_t strideB, const void* C, int64_t ldc, int64_t strideC,
                             void* D, int64_t ldd, int64_t strideD, int64_t M, int64_t N, int64_t K, int64_t batch,
                             float alpha, float beta, gemm_stream_t stream) {
    if ((a_major != GEMM_K_MAJOR && a_major != GEMM_MN_MAJOR) || (b_major != GEMM_K_MAJOR && b_major != GEMM_MN_MAJOR))
        return GEMM_ERR_INVALID_VALUE;
    Problem p = {M, N, K, batch, lda, ldb, ldc, ldd, strideA, strideB, strideC, strideD, beta, 0};
    p.a_mn = a_major == GEMM_MN_MAJOR ? 1 : 0;
    p.b_mn = b_major == GEMM_MN_MAJOR ? 1 : 0;
    p.acc16 = 1;
    return run(A, B, C, D, p, alpha, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_tn_f16_host(const void* A, int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc,
                               void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                               gemm_stream_t stream) {
    return run_host(A, lda, B, ldb, C, ldc, D, ldd, M, N, K, alpha, beta, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t score_softmax_stats_f16(const void* Q, int64_t ldq, int64_t strideQ, const void* K, int64_t ldk,
                                      int64_t strideK, float* row_max, float* row_sum, int64_t M, int64_t N, int64_t d,
                                      int64_t batch, float alpha, gemm_stream_t stream) {
    return run_softmax(Q, ldq, strideQ, K, ldk, strideK, row_max, row_sum, M, N, d, batch, alpha,
                       reinterpret_cast<cudaStream_t>(stream));
}

const char* gemm_status_string(gemm_status_t s) {
    switch (s) {
        case GEMM_OK: return "success";
        case GEMM_ERR_INVALID_VALUE: return "invalid value (size, leading dimension, stride, overlap or NULL pointer)";
        case GEMM_ERR_MISALIGNED: return "pointer not 2-byte aligned";
        case GEMM_ERR_UNSUPPORTED: return "unsupported device or problem size";
        case GEMM_ERR_CUDA: return "CUDA runtime or driver error";
        case GEMM_ERR_TIMEOUT: return "device-side wait timed out";
        case GEMM_ERR_WORKSPACE: return "scratch memory unavailable";
        case GEMM_ERR_BOUNDS: return "device-side bounds check failed (checked build)";
    }
    return "unknown status";
}

gemm_status_t gemm_tn_f16_last_device_error(void) {
    DeviceState* dev = nullptr;
    gemm_status_t st = device_state(&dev);
    if (st != GEMM_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t word = 0;
    if ((e = cudaMemcpy(&word, dev->err, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
    if (word != 0) {
        const uint32_t zero = 0;
        if ((e = cudaMemcpy(dev->err, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess) return cuda_fail(e);
        return (word >> 8) == 5u ? GEMM_ERR_TIMEOUT : (word >> 8) == 6u ? GEMM_ERR_BOUNDS : GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

int gemm_tn_f16_last_cuda_error(void) { return t_last_cuda_error; }

void gemm_tn_f16_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    int cur = 0;
    const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    for (int i = 0; i < kMaxDevices; ++i) {
        DeviceState& d = g_devices[i];
        if (d.ready && d.pool) {
            cudaSetDevice(i);
            cudaDeviceSynchronize();
            cudaMemPoolDestroy(d.pool);
            d.pool = nullptr;
            if (d.copy_in) cudaStreamDestroy(d.copy_in);
            if (d.copy_out) cudaStreamDestroy(d.copy_out);
            d.copy_in = d.copy_out = nullptr;
            d.ready = false;
        }
    }
    if (have_cur) cudaSetDevice(cur);
}

int gemm_tn_f16_version(void) { return 1 * 10000 + 0 * 100 + 0; }

int gemm_tn_f16_is_checked(void) { return kChecked ? 1 : 0; }

gemm_status_t gemm_tn_f16_plan(int64_t M, int64_t N, int64_t K, int64_t batch, int64_t lda, int64_t ldb, int64_t ldc,
                               int64_t ldd, int64_t strideA, int64_t strideB, int64_t strideC, int64_t strideD,
                               float beta, uint32_t align_flags, int32_t num_sms, gemm_tn_plan_t* plan) {
    if (!plan || num_sms <= 0) return GEMM_ERR_INVALID_VALUE;
    Problem p = {M, N, K, batch, lda, ldb, ldc, ldd, strideA, strideB, strideC, strideD, beta, align_flags};
    gemm_status_t st = validate(p);
    if (st != GEMM_OK) return st;
    Plan pl;
    make_plan(p, num_sms, pl);
    *plan = pl.pub;
    return GEMM_OK;
}

gemm_status_t gemm_tn_f16_set_option(int32_t option, int64_t value) {
    switch (option) {
        case GEMM_TN_OPT_WAIT_TIMEOUT_NS:
            if (value < 1000000 || value > 60000000000ll) return GEMM_ERR_INVALID_VALUE;
            g_opt_timeout_ns = value;
            return GEMM_OK;
        case GEMM_TN_OPT_SKIP_FIRST_LOAD: g_opt_skip_first_load = value ? 1 : 0; return GEMM_OK;
        case GEMM_TN_OPT_FORCE_BN:
            if (value != 0 && value != 128 && value != 256 && value != 432 && value != 512)
                return GEMM_ERR_INVALID_VALUE;
            g_opt_force_bn = value;
            return GEMM_OK;
        case GEMM_TN_OPT_FORCE_PAIR:
            if (value < 0 || value > 2) return GEMM_ERR_INVALID_VALUE;
            g_opt_force_pair = value;
            return GEMM_OK;
        case GEMM_TN_OPT_FORCE_SPLITS:
            if (value < 0 || value > 64) return GEMM_ERR_INVALID_VALUE;
            g_opt_force_splits = value;
            return GEMM_OK;
        case GEMM_TN_OPT_FORCE_SWAP:
            if (value < -1 || value > 1) return GEMM_ERR_INVALID_VALUE;
            g_opt_force_swap = value;
            return GEMM_OK;
        case GEMM_TN_OPT_FORCE_GENERIC_EPI: g_opt_force_generic = value ? 1 : 0; return GEMM_OK;
        case GEMM_TN_OPT_FORCE_PACK: g_opt_force_pack = value ? 1 : 0; return GEMM_OK;
        case GEMM_TN_OPT_STREAM_K:
            if (value < -1 || value > 1) return GEMM_ERR_INVALID_VALUE;
            g_opt_stream_k = value;
            return GEMM_OK;
        case GEMM_TN_OPT_GROUP_M:
            if (value < 0 || value > 64) return GEMM_ERR_INVALID_VALUE;
            g_opt_group_m = value;
            return GEMM_OK;
        case GEMM_TN_OPT_SERPENTINE:
            if (value < -1 || value > 1) return GEMM_ERR_INVALID_VALUE;
            g_opt_serpentine = value;
            return GEMM_OK;
        case GEMM_TN_OPT_ROW_LOADER: g_opt_row_loader = value ? 1 : 0; return GEMM_OK;
        case GEMM_TN_OPT_CHECK_TRIM_D:
            if (value < 0 || value > 4096) return GEMM_ERR_INVALID_VALUE;
            g_opt_check_trim_d = value;
            return GEMM_OK;
        case GEMM_TN_OPT_K_CLUSTER:
            if (value < -1 || value > 1) return GEMM_ERR_INVALID_VALUE;
            g_opt_k_cluster = value;
            return GEMM_OK;
        case GEMM_TN_OPT_SMALL:
            if (value != -1 && value != 0 && value != 1 && value != 64 && value != 128) return GEMM_ERR_INVALID_VALUE;
            g_opt_small = value;
            return GEMM_OK;

    }
    return GEMM_ERR_INVALID_VALUE;
}

int64_t gemm_tn_f16_get_option(int32_t option) {
    switch (option) {
        case GEMM_TN_OPT_WAIT_TIMEOUT_NS: return g_opt_timeout_ns.load();
        case GEMM_TN_OPT_SKIP_FIRST_LOAD: return g_opt_skip_first_load.load();
        case GEMM_TN_OPT_FORCE_BN: return g_opt_force_bn.load();
        case GEMM_TN_OPT_FORCE_PAIR: return g_opt_force_pair.load();
        case GEMM_TN_OPT_FORCE_SPLITS: return g_opt_force_splits.load();
        case GEMM_TN_OPT_FORCE_SWAP: return g_opt_force_swap.load();
        case GEMM_TN_OPT_FORCE_GENERIC_EPI: return g_opt_force_generic.load();
        case GEMM_TN_OPT_FORCE_PACK: return g_opt_force_pack.load();
        case GEMM_TN_OPT_STREAM_K: return g_opt_stream_k.load();
        case GEMM_TN_OPT_GROUP_M: return g_opt_group_m.load();
        case GEMM_TN_OPT_SERPENTINE: return g_opt_serpentine.load();
        case GEMM_TN_OPT_ROW_LOADER: return g_opt_row_loader.load();
        case GEMM_TN_OPT_CHECK_TRIM_D: return g_opt_check_trim_d.load();
        case GEMM_TN_OPT_K_CLUSTER: return g_opt_k_cluster.load();
        case GEMM_TN_OPT_SMALL: return g_opt_small.load();

    }
    return -1;
}

}  // extern "C"
