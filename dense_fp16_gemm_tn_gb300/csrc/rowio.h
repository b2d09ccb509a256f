// Row segments of 64 fp16 elements at any 2-byte alignment, moved through the
// 16-byte-aligned words that cover them.  The epilogue uses these for C and D rows
// whose start or leading dimension rules out TMA (tensor copies need 16-byte-aligned
// rows): every access is a whole aligned word, except the stores to the two edge words
// of a segment, which go out in smaller aligned pieces so that no byte outside the
// segment is written.  Plain C++ off the device, so that the index arithmetic is tested on the
// host.
#pragma once

#include <cstdint>
#include <cstring>

#ifdef __CUDACC__
#define GTN_ROWIO __host__ __device__ __forceinline__
#else
#define GTN_ROWIO inline
#endif

namespace gtn {

// Checker of a row segment [a, b) (byte addresses) before it is read or written: the
// default accepts everything; the checked build passes one that tests the range against
// the matrix's extent (checked.h).  A rejected segment is neither read nor written.
struct NoCheck {
    GTN_ROWIO bool operator()(uintptr_t, uintptr_t) const { return true; }
};

// (lo >> 16) | (hi << 16): the upper half of lo followed by the lower half of hi.
GTN_ROWIO uint32_t join_halves(uint32_t lo, uint32_t hi) { return (lo >> 16) | (hi << 16); }

GTN_ROWIO void load_word16(uintptr_t addr, uint32_t* w) {
#ifdef __CUDA_ARCH__
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(addr));
    w[0] = x.x;
    w[1] = x.y;
    w[2] = x.z;
    w[3] = x.w;
#else
#ifdef GTN_ROWIO_TRACE
    GTN_ROWIO_TRACE(addr);  // host tests record which words are read
#endif
    std::memcpy(w, reinterpret_cast<const void*>(addr), 16);
#endif
}

GTN_ROWIO void store_word16(uintptr_t addr, const uint32_t* w) {
#ifdef __CUDA_ARCH__
    *reinterpret_cast<uint4*>(addr) = make_uint4(w[0], w[1], w[2], w[3]);
#else
    std::memcpy(reinterpret_cast<void*>(addr), w, 16);
#endif
}

// Bytes [lo, hi) (even offsets, lo < hi <= 16) of the aligned 16-byte word at `wa`,
// whose content is w0..w3, in at most three naturally aligned 2-, 4- or 8-byte stores
// (a 2-byte piece up to 4-byte alignment, a 4-byte piece up to 8, an 8-byte piece, then
// 4- and 2-byte pieces down to hi).
GTN_ROWIO void store_part16(uintptr_t wa, uint32_t lo, uint32_t hi, uint32_t w0, uint32_t w1, uint32_t w2,
                            uint32_t w3) {
    auto word = [&](uint32_t o) { return (o & 8u) ? ((o & 4u) ? w3 : w2) : ((o & 4u) ? w1 : w0); };
    auto put16 = [&](uint32_t o) {
        const uint16_t v = static_cast<uint16_t>(word(o) >> (8u * (o & 2u)));
#ifdef __CUDA_ARCH__
        *reinterpret_cast<uint16_t*>(wa + o) = v;
#else
        std::memcpy(reinterpret_cast<void*>(wa + o), &v, 2);
#endif
    };
    auto put32 = [&](uint32_t o) {
        const uint32_t v = word(o);
#ifdef __CUDA_ARCH__
        *reinterpret_cast<uint32_t*>(wa + o) = v;
#else
        std::memcpy(reinterpret_cast<void*>(wa + o), &v, 4);
#endif
    };
    auto put64 = [&](uint32_t o) {
        const uint32_t a = (o & 8u) ? w2 : w0, b = (o & 8u) ? w3 : w1;
#ifdef __CUDA_ARCH__
        *reinterpret_cast<uint2*>(wa + o) = make_uint2(a, b);
#else
        const uint32_t v[2] = {a, b};
        std::memcpy(reinterpret_cast<void*>(wa + o), v, 8);
#endif
    };
    uint32_t o = lo;
    if ((o & 2u) && o + 2u <= hi) { put16(o); o += 2u; }
    if ((o & 4u) && o + 4u <= hi) { put32(o); o += 4u; }
    if (!(o & 7u) && o + 8u <= hi) { put64(o); o += 8u; }
    if (o + 4u <= hi) { put32(o); o += 4u; }
    if (o + 2u <= hi) { put16(o); o += 2u; }
}

// The nine aligned words that cover halves src[0..63].  Only words holding at least one
// of the first `valid` halves are read (so no read leaves the pages those elements live
// on); the others are zero.  Returns the offset of src in its first word, in halves.
// The segment [src, src + valid) goes through `chk` first; if it is rejected nothing is
// read and all nine words are zero.
template <class Chk = NoCheck>
GTN_ROWIO uint32_t load_cover64(const uint16_t* src, int valid, uint32_t (&v)[36], const Chk& chk = Chk()) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(src);
    const uintptr_t base = a & ~uintptr_t(15);
    const bool any = valid > 0 && chk(a, a + 2u * static_cast<uint32_t>(valid));
    const uintptr_t end = a + 2u * static_cast<uint32_t>(any ? valid : 0);
#pragma unroll
    for (int q = 0; q < 9; ++q) {
        const uintptr_t wa = base + 16u * q;
        uint32_t* w = v + 4 * q;
        if (any && wa < end) {
            load_word16(wa, w);
        } else {
            w[0] = w[1] = w[2] = w[3] = 0u;
        }
    }
    return static_cast<uint32_t>(a - base) >> 1;
}

// The 64 halves starting `sh` (0..7) halves into the covering words, as 32 words of two
// halves (low half first): selects by two and by one words, then a one-half shift for
// an odd `sh`.  The same instructions for every `sh`: no divergence, no indexed registers.
GTN_ROWIO void align_cover64(const uint32_t (&v)[36], uint32_t sh, uint32_t (&w)[32]) {
    const bool by2 = (sh & 4u) != 0, by1 = (sh & 2u) != 0, odd = (sh & 1u) != 0;
    uint32_t t[34];
#pragma unroll
    for (int i = 0; i < 34; ++i) t[i] = by2 ? v[i + 2] : v[i];
    uint32_t u[33];
#pragma unroll
    for (int i = 0; i < 33; ++i) u[i] = by1 ? t[i + 1] : t[i];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = odd ? join_halves(u[i], u[i + 1]) : u[i];
}

// The mirror of align_cover64: the 64 halves in o (32 words, low half first) placed at
// an offset of `sh` (0..7) halves into nine 16-byte words z (zero elsewhere).
GTN_ROWIO void place_row64(uint32_t sh, const uint32_t (&o)[32], uint32_t (&z)[36]) {
    const bool by2 = (sh & 4u) != 0, by1 = (sh & 2u) != 0, odd = (sh & 1u) != 0;
    uint32_t op[33];  // one half to the right when sh is odd
#pragma unroll
    for (int j = 0; j < 33; ++j) {
        const uint32_t lo = j > 0 ? o[j - 1] : 0u, hi = j < 32 ? o[j] : 0u;
        op[j] = odd ? join_halves(lo, hi) : hi;
    }
    uint32_t t[34];
#pragma unroll
    for (int i = 0; i < 34; ++i) t[i] = by1 ? (i >= 1 ? op[i - 1] : 0u) : (i < 33 ? op[i] : 0u);
#pragma unroll
    for (int i = 0; i < 36; ++i) z[i] = by2 ? (i >= 2 ? t[i - 2] : 0u) : (i < 34 ? t[i] : 0u);
}

// Writes the first `valid` (0..64) of the 64 halves in o (32 words, low half first) to
// dst: place_row64 puts them in the covering words; whole words go out as 16-byte
// stores, the two edge words in aligned pieces (store_part16).
// The segment [dst, dst + valid) goes through `chk` first; if it is rejected nothing is
// written.
template <class Chk = NoCheck>
GTN_ROWIO void store_row64(uint16_t* dst, int valid, const uint32_t (&o)[32], const Chk& chk = Chk()) {
    if (valid <= 0) return;
    const uintptr_t a = reinterpret_cast<uintptr_t>(dst);
    const uintptr_t base = a & ~uintptr_t(15);
    const uintptr_t end = a + 2u * static_cast<uint32_t>(valid);
    if (!chk(a, end)) return;
    uint32_t z[36];
    place_row64(static_cast<uint32_t>(a - base) >> 1, o, z);
#pragma unroll
    for (int q = 0; q < 9; ++q) {
        const uintptr_t wa = base + 16u * q;
        if (wa >= end) break;
        if (wa >= a && wa + 16u <= end) {
            store_word16(wa, z + 4 * q);
        } else {
            const uint32_t lo = a > wa ? static_cast<uint32_t>(a - wa) : 0u;
            const uint32_t hi = end < wa + 16u ? static_cast<uint32_t>(end - wa) : 16u;
            store_part16(wa, lo, hi, z[4 * q], z[4 * q + 1], z[4 * q + 2], z[4 * q + 3]);
        }
    }
}

}  // namespace gtn
