// gemm_tn_f16_splitk_static: the split-K GEMM with its scratch memory built
// into the library, so that a call allocates no device memory at all.
//
// Who needs it: callers that may not allocate device memory at the moment they
// call the GEMM.  Examples are a caching allocator or memory-pool
// implementation that calls the GEMM from code holding its own lock (calling
// cudaMalloc there would re-enter the allocator or deadlock), and services
// that reserve their whole device-memory budget at start-up and forbid
// allocation on the request path (cudaMalloc can synchronise the device and
// has no latency bound).  The regular entry points take their split-K scratch
// from a stream-ordered pool; this one never calls cudaMalloc, cudaFree or any
// allocating routine.
//
// The scratch is one file-scope device array of GEMM_TN_STATIC_SCRATCH_BYTES,
// present on every GPU that loads the library until the process exits.  Host
// code must not pass the array's name to a kernel (on the host it is only a
// stand-in symbol); its device address is looked up once per device with
// cudaGetSymbolAddress and cached.  Every call on a device shares the array,
// so calls whose work can overlap on the GPU (e.g. on two unsynchronised
// streams) race on it.  Nothing in it has to start at zero: each K slice's
// epilogue writes every partial sum of its tile before the reduction reads it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "gemm_tn_f16.h"
#include "internal.h"

namespace gtn {
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[GEMM_TN_STATIC_SCRATCH_BYTES];

struct StaticDevice {
    bool ready = false;
    int sms = 0;
    float* scratch = nullptr;  // device address of g_static_scratch on this device
    uint32_t* err = nullptr;   // device address of the library's error word
};

constexpr int kMaxDev = 64;
StaticDevice g_static_dev[kMaxDev];
std::mutex g_static_mu;

// One-time set-up per device, run with that device current.
gemm_status_t static_device(StaticDevice** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDev) return GEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_static_mu);
    StaticDevice& d = g_static_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (!(major == 10 && minor == 3)) return GEMM_ERR_UNSUPPORTED;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return GEMM_ERR_CUDA;
        d.scratch = static_cast<float*>(p);
        if (error_word_address(&d.err) != cudaSuccess) return GEMM_ERR_CUDA;
        d.ready = true;
    }
    *out = &d;
    return GEMM_OK;
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    });
    return fn;
}

// 2-D operand (rows x K, leading dimension ld) as a 3-D map with batch extent 1.
bool operand_map(CUtensorMap* m, const void* base, int64_t K, int64_t rows, int64_t ld, uint32_t box_rows) {
    EncodeFn fn = encoder();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows), 1};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2u, static_cast<cuuint64_t>(ld * rows) * 2u};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool overlap(const void* a, int64_t an, const void* b, int64_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(bn) && b0 < a0 + static_cast<uintptr_t>(an);
}

}  // namespace
}  // namespace gtn

using namespace gtn;

extern "C" GEMM_TN_API gemm_status_t gemm_tn_f16_splitk_static(const void* A, int64_t lda, const void* B, int64_t ldb,
                                                               const void* C, int64_t ldc, void* D, int64_t ldd,
                                                               int64_t M, int64_t N, int64_t K, float alpha,
                                                               float beta, int32_t splits, gemm_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    // ---- argument checks (same rules as gemm_tn_f16)
    if (M < 0 || N < 0 || K < 0 || splits < 0) return GEMM_ERR_INVALID_VALUE;
    const int64_t lim = int64_t(1) << 31;
    if (M >= lim || N >= lim || K >= lim) return GEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!D || ldd < N) return GEMM_ERR_INVALID_VALUE;
    if (K > 0 && (!A || !B || lda < K || ldb < K)) return GEMM_ERR_INVALID_VALUE;
    if (beta != 0.0f && (!C || ldc < N)) return GEMM_ERR_INVALID_VALUE;
    auto odd = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) != 0; };
    if (odd(D) || (beta != 0.0f && odd(C))) return GEMM_ERR_MISALIGNED;
    const int64_t d_bytes = 2 * ((M - 1) * ldd + N);
    if (K > 0 && (overlap(D, d_bytes, A, 2 * ((M - 1) * lda + K)) || overlap(D, d_bytes, B, 2 * ((N - 1) * ldb + K))))
        return GEMM_ERR_INVALID_VALUE;
    if (beta != 0.0f && C != D && overlap(D, d_bytes, C, 2 * ((M - 1) * ldc + N))) return GEMM_ERR_INVALID_VALUE;
    if (beta != 0.0f && C == D && ldc != ldd) return GEMM_ERR_INVALID_VALUE;
    // No scratch for a repacked copy: operands must be fetchable by TMA as they are.
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (K > 0 && (!al16(A) || !al16(B) || lda % 8 != 0 || ldb % 8 != 0)) return GEMM_ERR_MISALIGNED;

    StaticDevice* dev = nullptr;
    gemm_status_t st = static_device(&dev);
    if (st != GEMM_OK) return st;
    // byte ranges for the checked build's device-side bounds checks
    auto ext = [](const void* b, int64_t bytes) {
        const uint64_t lo = static_cast<uint64_t>(reinterpret_cast<uintptr_t>(b));
        return Extent{lo, lo + static_cast<uint64_t>(bytes)};
    };
    ReduceChecks chk = {};
    chk.c = beta != 0.0f ? ext(C, 2 * ((M - 1) * ldc + N)) : Extent{};
    chk.d = ext(D, d_bytes);
    chk.err = dev->err;
    if (K == 0) {
        return launch_scale(M, N, 1, beta, C, ldc, 0, D, ldd, 0, dev->sms, stream, chk) == cudaSuccess
                   ? GEMM_OK
                   : GEMM_ERR_CUDA;
    }

    // ---- plan: split-K over 128-row tiles; operands swapped when M is small
    const bool swap = M <= 64 && N >= 128 && N >= 2 * M;
    const int bn = swap ? (M <= 16 ? 16 : M <= 32 ? 32 : 64) : 128;
    const int64_t rows_a = swap ? N : M, rows_b = swap ? M : N;
    const int64_t tiles = cdiv(rows_a, 128) * cdiv(rows_b, bn);
    const int64_t kb = cdiv(K, 64);
    int64_t s = splits;
    if (s == 0) {
        // This path's own rule (the pooled entry points plan differently, with stream-K and
        // data-parallel tiles as alternatives): the fewest K slices, up to 64 of at least four
        // k-blocks, that minimise waves x (slice length + 2).  With a wave or more of tiles that
        // is one slice, whose fp32 result still passes through the array and the sum kernel.
        int64_t best = INT64_MAX;
        s = 1;
        const int64_t max_s = kb / 4 < 64 ? (kb / 4 < 1 ? 1 : kb / 4) : 64;
        for (int64_t c = 1; c <= max_s; ++c) {
            const int64_t cost = cdiv(tiles * c, dev->sms) * (cdiv(kb, c) + 2);
            if (cost < best) { best = cost; s = c; }
        }
    }
    if (s > kb) s = kb;
    if (s * M * N * 4 > static_cast<int64_t>(GEMM_TN_STATIC_SCRATCH_BYTES)) return GEMM_ERR_WORKSPACE;

    TcVariant v;
    if (!find_tc_variant(bn, 1, swap ? EPI_PARTIAL_SWAP : EPI_PARTIAL, 0, &v)) return GEMM_ERR_UNSUPPORTED;
    CUtensorMap mapA, mapB;
    // MMA A operand: the 128-row side; MMA B operand: the BN-row side.
    if (!operand_map(&mapA, swap ? B : A, K, rows_a, swap ? ldb : lda, 128) ||
        !operand_map(&mapB, swap ? A : B, K, rows_b, swap ? lda : ldb, static_cast<uint32_t>(bn)))
        return GEMM_ERR_UNSUPPORTED;

    KParams kp;
    std::memset(&kp, 0, sizeof(kp));
    kp.rows_a = static_cast<int32_t>(rows_a);
    kp.rows_b = static_cast<int32_t>(rows_b);
    kp.K = static_cast<int32_t>(K);
    kp.batch = 1;
    kp.tiles_m = static_cast<int32_t>(cdiv(rows_a, 128));
    kp.tiles_n = static_cast<int32_t>(cdiv(rows_b, bn));
    kp.splits = static_cast<int32_t>(s);
    kp.kb_total = static_cast<int32_t>(kb);
    kp.group_m = 16;
    kp.num_units = tiles * s;
    kp.M = static_cast<int32_t>(M);
    kp.N = static_cast<int32_t>(N);
    kp.alpha = alpha;
    kp.beta = beta;
    kp.D = D;
    kp.ldd = ldd;
    kp.C = C;
    kp.ldc = ldc;
    kp.W = dev->scratch;
    kp.err = dev->err;
    kp.timeout_ns = 2000000000ull;
    kp.ext_a = ext(swap ? B : A, 2 * ((rows_a - 1) * (swap ? ldb : lda) + K));
    kp.ext_b = ext(swap ? A : B, 2 * ((rows_b - 1) * (swap ? lda : ldb) + K));
    kp.ext_c = chk.c;
    kp.ext_d = chk.d;
    kp.ext_w = ext(dev->scratch, s * M * N * 4);
    chk.w = kp.ext_w;

    int64_t grid = 0;
    if (launch_tc_variant(v, mapA, mapB, mapA, mapA, kp, dev->sms, stream, &grid) != cudaSuccess) return GEMM_ERR_CUDA;
    if (launch_splitk_reduce(dev->scratch, static_cast<int32_t>(s), M, N, 1, alpha, beta, C, ldc, 0, D, ldd, 0,
                             dev->sms, stream, chk) != cudaSuccess)
        return GEMM_ERR_CUDA;
    return GEMM_OK;
}
