// Device-side bounds checks of the checked build (the library compiled with
// -DGTN_CHECKED, libgemm_tn_f16_checked.so).  In that build every global-memory
// access the kernels make with their own loads and stores -- the row-word loads and
// stores of C and D, the predicated element accesses, the row loader's operand
// reads, the repack, the split-K sum and the K == 0 scale -- is first checked against
// the byte range of the matrix it belongs to.  An access outside it is skipped, and
// the first one recorded in the device error word as 0x600 | site, which
// gemm_tn_f16_last_device_error() reports as GEMM_ERR_BOUNDS.  Tensor copies (TMA)
// are bounded by their tensor maps and are not checked here.  In the regular build
// the checks compile to nothing.
#pragma once

#include <cstdint>

namespace gtn {

#ifdef GTN_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// Byte range [lo, hi) of one matrix as the caller passed it.
struct Extent {
    uint64_t lo, hi;
};

// Sites recorded in the low byte of the error word.
enum CheckSite : uint32_t {
    CHK_EPI_C_ROW = 0x01,     // epilogue: C row words (misaligned C)
    CHK_EPI_D_ROW = 0x02,     // epilogue: D row words (misaligned D)
    CHK_RL_A = 0x03,          // row loader: A rows
    CHK_RL_B = 0x04,          // row loader: B rows
    CHK_EPI_C_ELEM = 0x05,    // predicated / swapped epilogue: C elements
    CHK_EPI_D_ELEM = 0x06,    // predicated / swapped epilogue: D elements
    CHK_EPI_W = 0x07,         // split-K partial sums written by the GEMM
    CHK_REPACK_SRC = 0x08,    // repack: source row groups
    CHK_REPACK_DST = 0x09,    // repack: destination groups
    CHK_REDUCE_W = 0x0a,      // split-K sum: partial sums read
    CHK_REDUCE_C = 0x0b,      // split-K sum and scale: C read
    CHK_REDUCE_D = 0x0c,      // split-K sum and scale: D written
};

#ifdef __CUDACC__
// True when [a, b) lies inside e; otherwise records the site (first violation only).
__device__ __forceinline__ bool in_extent(uint64_t a, uint64_t b, const Extent& e, uint32_t* err, uint32_t site) {
    if (a <= b && a >= e.lo && b <= e.hi) return true;
    if (err) atomicCAS(err, 0u, 0x600u | site);
    return false;
}

// Range check usable as the row-word helpers' checker (rowio.h): in the regular build
// it is never instantiated with kChecked false at the call sites that pass it.
struct DevCheck {
    Extent e;
    uint32_t* err;
    uint32_t site;
    __device__ __forceinline__ bool operator()(uintptr_t a, uintptr_t b) const {
        return in_extent(static_cast<uint64_t>(a), static_cast<uint64_t>(b), e, err, site);
    }
};

// One element at ptr: checked in the checked build, always accepted otherwise.
template <class T>
__device__ __forceinline__ bool chk_elem(const T* ptr, const Extent& e, uint32_t* err, uint32_t site) {
    if constexpr (kChecked) {
        const uint64_t a = static_cast<uint64_t>(reinterpret_cast<uintptr_t>(ptr));
        return in_extent(a, a + sizeof(T), e, err, site);
    } else {
        return true;
    }
}
#endif

// The row-word helpers' checker for a matrix: DevCheck in the checked build, else none.
#ifdef GTN_CHECKED
#define GTN_ROW_CHECK(ext, err, site) ::gtn::DevCheck{(ext), (err), (site)}
#else
#define GTN_ROW_CHECK(ext, err, site) ::gtn::NoCheck{}
#endif

}  // namespace gtn
