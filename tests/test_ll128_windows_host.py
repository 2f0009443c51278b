"""Index arithmetic of the LL128 lane windows, checked on the CPU.

A lane of an LL128 line (63 16-bit or 31 32-bit payload elements, the
count flag in element 0 of lane 0: "Every Microsecond Matters", technique
4) carries a 16-byte window that starts one element before a lane
boundary. The kernels read such a window with two aligned 16-byte loads
shifted into place and write it with a few aligned stores
(`ll128_gather_fast`, `ll128_scatter_fast`); windows at the edge of a
segment or of the message go element by element. This test compiles those
helpers, exactly as they stand in the kernel source, for the host with g++
(a small shim supplies the CUDA types and `__byte_perm`), and checks on
every window of many message shapes that:

* the fast and element-by-element paths gather the same words and write
  the same bytes, into a whole-message output and into a segment output;
* the fast path reads only inside the message and writes nothing outside;
* scattering every window reproduces the message exactly.
"""

import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KERNELS = os.path.join(ROOT, "tp_allreduce_persistent_b300", "csrc", "llar_kernels.cu")

SHIM = r"""
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <random>
#include <vector>
#define __device__
#define __forceinline__ inline
struct uint4 { unsigned x, y, z, w; };
static inline uint4 make_uint4(unsigned a, unsigned b, unsigned c, unsigned d) { return {a, b, c, d}; }
using std::min;
// byte permute: result byte i = byte (s >> 4i) & 7 of {y:x}
static inline unsigned __byte_perm(unsigned x, unsigned y, unsigned s) {
  unsigned char b[8];
  memcpy(b, &x, 4);
  memcpy(b + 4, &y, 4);
  unsigned r = 0;
  for (int i = 0; i < 4; ++i) r |= (unsigned)b[(s >> (4 * i)) & 7] << (8 * i);
  return r;
}
template <int DT> struct Fmt;
template <> struct Fmt<0> {
  static constexpr int kBytes = 4;
  static unsigned load(const char* b, size_t i) { unsigned v; memcpy(&v, b + i * 4, 4); return v; }
  static void store(char* b, size_t i, unsigned v) { memcpy(b + i * 4, &v, 4); }
};
template <> struct Fmt<2> {
  static constexpr int kBytes = 2;
  static unsigned load(const char* b, size_t i) { unsigned short v; memcpy(&v, b + i * 2, 2); return v; }
  static void store(char* b, size_t i, unsigned v) { unsigned short h = (unsigned short)v; memcpy(b + i * 2, &h, 2); }
};
template <int DT> unsigned word_elem(unsigned w, int k) {
  return Fmt<DT>::kBytes == 4 ? w : (w >> (16 * k)) & 0xFFFFu;
}
"""

MAIN = r"""
static const int kGuard = 64;  // bytes around every buffer (a multiple of 16)
template <int DT> int run(size_t count, int N, std::mt19937& rng) {
  constexpr int EB = Fmt<DT>::kBytes, P = 128 / EB - 1;
  const size_t nbytes = count * EB;
  std::vector<char> in(nbytes + 2 * kGuard);
  for (auto& c : in) c = (char)rng();
  const char* src = in.data() + kGuard;
  const size_t seg = (count + N - 1) / N, L = (seg + P - 1) / P;
  std::vector<char> o1(nbytes + 2 * kGuard, 0x55), o2(nbytes + 2 * kGuard, 0x55);
  int bad = 0;
  for (int s = 0; s < N; ++s) {
    const size_t lo = std::min(count, (size_t)s * seg), hi = std::min(count, lo + seg);
    std::vector<char> r1((hi - lo) * EB + 2 * kGuard, 0x33), r2((hi - lo) * EB + 2 * kGuard, 0x33);
    for (size_t l = 0; l < L; ++l)
      for (int j = 0; j < 8; ++j) {
        unsigned wf[4] = {1, 2, 3, 4}, ws[4] = {0, 0, 0, 0};
        const bool af = ll128_gather<DT>(src, count, seg, s, l, j, wf);
        const bool as = ll128_gather_slow<DT>(src, count, seg, s, l, j, ws);
        size_t first;
        if (ll128_window<DT>(count, seg, s, l, j, first)) {
          const size_t off = first * EB, vb = off & ~(size_t)15;
          const unsigned h = (unsigned)(off & 15) >> 1;
          if (off + 16 > nbytes) ++bad;                                  // window past the message
          if (!(h != 0 && vb + 32 > nbytes) && vb + (h ? 32 : 16) > nbytes) ++bad;  // fast read past it
        }
        if (af != as || (as && memcmp(wf, ws, 16) != 0)) ++bad;
        if (!as) continue;
        ll128_scatter<DT>(o1.data() + kGuard, 0, count, seg, s, l, j, ws);
        ll128_scatter_slow<DT>(o2.data() + kGuard, 0, count, seg, s, l, j, ws);
        ll128_scatter<DT>(r1.data() + kGuard, lo, count, seg, s, l, j, ws);
        ll128_scatter_slow<DT>(r2.data() + kGuard, lo, count, seg, s, l, j, ws);
      }
    if (r1 != r2) ++bad;
    if (memcmp(r2.data() + kGuard, src + lo * EB, (hi - lo) * EB) != 0) ++bad;
  }
  if (o1 != o2) ++bad;  // guards included: nothing written outside
  if (memcmp(o2.data() + kGuard, src, nbytes) != 0) ++bad;
  if (bad) printf("mismatch: %d-byte elements, count %zu, %d ranks\n", EB, count, N);
  return bad;
}
int main() {
  std::mt19937 rng(1);
  std::vector<size_t> counts = {1, 2, 7, 8, 9, 62, 63, 64, 65, 126, 127, 128, 129, 500, 1001, 4096, 8191, 8193, 65537};
  for (int k = 0; k < 20; ++k) counts.push_back(1 + rng() % 200000);
  int bad = 0;
  for (size_t c : counts)
    for (int N = 2; N <= 8; ++N) bad += run<0>(c, N, rng) + run<2>(c, N, rng);
  printf("bad %d\n", bad);
  return bad != 0;
}
"""


def _helpers():
    src = open(KERNELS).read()
    start = re.search(r"template <int DT>\n__device__ __forceinline__ bool ll128_window\(", src)
    end = re.search(r"template <int DT>\n__device__ __forceinline__ void body_ll128\(", src)
    assert start and end and start.start() < end.start(), "LL128 window helpers not found in the kernel source"
    return src[start.start():end.start()]


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_ll128_windows_fast_path_equals_element_path(tmp_path):
    cpp = tmp_path / "windows.cpp"
    cpp.write_text(SHIM + _helpers() + MAIN)
    exe = tmp_path / "windows"
    subprocess.run(["g++", "-O1", "-std=c++17", "-o", str(exe), str(cpp)], check=True,
                   capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and "bad 0" in out.stdout, out.stdout + out.stderr


# plausible mistakes, each planted in a host copy of the helpers: the check
# above must fail on every one of them
MUTATIONS = {
    "byte permutation": ("0x5432", "0x5410"),
    "two-word shift": ("x[i] = x[i + 2]", "x[i] = x[i + 1]"),
    "lane-0 flag element": ("if (!skip0 && (first & 7) == 0)", "if ((first & 7) == 0)"),
    "segment bound": ("sl0 + V - 1 <= lim", "sl0 + V - 2 <= lim"),
}


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_ll128_window_check_catches_planted_mistakes(name, tmp_path):
    old, new = MUTATIONS[name]
    helpers = _helpers()
    assert old in helpers, name
    cpp = tmp_path / "mutant.cpp"
    cpp.write_text(SHIM + helpers.replace(old, new, 1) + MAIN)
    exe = tmp_path / "mutant"
    subprocess.run(["g++", "-O1", "-std=c++17", "-o", str(exe), str(cpp)], check=True,
                   capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode != 0 and "bad 0" not in out.stdout, name
