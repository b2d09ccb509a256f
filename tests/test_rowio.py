"""The epilogue's access to C and D rows at any 2-byte alignment (csrc/rowio.h),
compiled for the host with g++: for every offset of the row in its 16-byte word and
every length 0..64, stores write exactly the row's elements (guard bytes around them
untouched), loads read only whole aligned words that hold at least one of the row's
elements, and the realigned values are the row's values; a load at one alignment and a
store at another move a row unchanged; the checker hook of the checked build sees the
row segment and, when it rejects it, nothing is read or written."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "dense_fp16_gemm_tn_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <vector>
static std::vector<uintptr_t> g_reads;
static void trace(uintptr_t a) { g_reads.push_back(a); }
#define GTN_ROWIO_TRACE(a) trace(a)
#include "rowio.h"
using namespace gtn;

alignas(64) static uint16_t buf[1024];
alignas(64) static uint16_t src[1024];
static long bad = 0, cases = 0;
#define CHECK(c, ...) do { if (!(c)) { if (bad < 20) { std::printf(__VA_ARGS__); std::printf("\n"); } ++bad; } } while (0)

int main() {
    for (int i = 0; i < 1024; ++i) src[i] = static_cast<uint16_t>(0x3000 + i * 7);
    uint32_t o[32];
    for (int i = 0; i < 32; ++i) o[i] = (uint32_t(0x1000 + 2 * i + 1) << 16) | uint32_t(0x1000 + 2 * i);
    for (int off = 64; off < 64 + 24; ++off) {          // every position in a 16-byte word, several words
        for (int valid = 0; valid <= 64; ++valid) {
            ++cases;
            // store: exactly [off, off + valid) changes
            for (int i = 0; i < 1024; ++i) buf[i] = 0xAAAA;
            store_row64(buf + off, valid, o);
            for (int i = 0; i < 1024; ++i) {
                const bool in = i >= off && i < off + valid;
                const uint16_t want = in ? static_cast<uint16_t>(0x1000 + (i - off)) : 0xAAAA;
                CHECK(buf[i] == want, "store off %d valid %d: buf[%d] = %04x want %04x", off, valid, i, buf[i], want);
            }
            // load: only words holding a real element are read; values realigned
            g_reads.clear();
            uint32_t v[36], w[32];
            const uint32_t sh = load_cover64(src + off, valid, v);
            CHECK(sh == static_cast<uint32_t>(off % 8), "shift off %d: %u", off, sh);
            const uintptr_t a = reinterpret_cast<uintptr_t>(src + off), e = a + 2u * valid;
            for (uintptr_t r : g_reads) {
                CHECK(r % 16 == 0, "unaligned read");
                CHECK(r < e && r + 16 > a, "load off %d valid %d reads a word with no element of the row", off, valid);
            }
            // every word that holds an element is read
            size_t need = 0;
            for (uintptr_t r = a & ~uintptr_t(15); valid > 0 && r < e; r += 16) ++need;
            CHECK(g_reads.size() == need, "load off %d valid %d: %zu reads, want %zu", off, valid, g_reads.size(), need);
            align_cover64(v, sh, w);
            for (int k = 0; k < valid; ++k) {
                const uint16_t got = static_cast<uint16_t>(w[k >> 1] >> (16 * (k & 1)));
                CHECK(got == src[off + k], "load off %d valid %d: element %d = %04x want %04x", off, valid, k, got, src[off + k]);
            }
            // round trip to another alignment
            const int off2 = 200 + (off * 5) % 16;
            for (int i = 0; i < 1024; ++i) buf[i] = 0x5555;
            store_row64(buf + off2, valid, w);
            for (int i = 0; i < 1024; ++i) {
                const bool in = i >= off2 && i < off2 + valid;
                const uint16_t want = in ? src[off + (i - off2)] : 0x5555;
                CHECK(buf[i] == want, "round trip off %d -> %d valid %d: buf[%d]", off, off2, valid, i);
            }
        }
    }
    // the checker hook of the checked build: it sees exactly the row segment, and a
    // rejected segment is neither read nor written
    struct Rec {
        bool accept;
        mutable uintptr_t lo = 0, hi = 0;
        bool operator()(uintptr_t a, uintptr_t b) const { lo = a; hi = b; return accept; }
    };
    for (int off = 64; off < 64 + 16; ++off) {
        for (int valid = 1; valid <= 64; valid += 9) {
            for (int acc = 0; acc < 2; ++acc) {
                ++cases;
                Rec chk{acc != 0};
                g_reads.clear();
                uint32_t v[36];
                load_cover64(src + off, valid, v, chk);
                const uintptr_t a = reinterpret_cast<uintptr_t>(src + off);
                CHECK(chk.lo == a && chk.hi == a + 2u * valid, "checker saw the wrong load segment");
                if (!acc) {
                    CHECK(g_reads.empty(), "rejected load off %d valid %d still read memory", off, valid);
                    bool zero = true;
                    for (int q = 0; q < 36; ++q) zero = zero && v[q] == 0;
                    CHECK(zero, "rejected load returned data");
                }
                for (int i = 0; i < 1024; ++i) buf[i] = 0xAAAA;
                Rec chk2{acc != 0};
                store_row64(buf + off, valid, o, chk2);
                const uintptr_t d = reinterpret_cast<uintptr_t>(buf + off);
                CHECK(chk2.lo == d && chk2.hi == d + 2u * valid, "checker saw the wrong store segment");
                int changed = 0;
                for (int i = 0; i < 1024; ++i) changed += buf[i] != 0xAAAA;
                CHECK(changed == (acc ? valid : 0), "store off %d valid %d accept %d changed %d", off, valid, acc, changed);
            }
        }
    }
    std::printf("cases %ld bad %ld\n", cases, bad);
    return bad == 0 ? 0 : 1;
}
"""


def test_row_segments_at_any_alignment(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no g++")
    src = tmp_path / "rowio.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "rowio"
    subprocess.run([gxx, "-O1", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "bad 0" in out.stdout, out.stdout
