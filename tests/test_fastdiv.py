"""The multiply-shift division by invariant integers the decode attention uses
for its stream-K piece arithmetic (csrc/internal.h: make_fastdiv, fast_div),
compiled for the host and checked against plain integer division: every
divisor up to 3000 with dividends at and around its multiples, divisors
spread over [1, 2^31), and the extreme dividends 0 and 2^32 - 1."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "megatron_tensor_layers_tp_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include "internal.h"
using namespace tpk;
static int bad = 0;
static void check(uint32_t n, uint32_t d, const FastDiv& f) {
  if (fast_div(n, f) != n / d) {
    if (bad < 5) std::printf("mismatch n=%u d=%u got=%u want=%u\n", n, d, fast_div(n, f), n / d);
    ++bad;
  }
}
int main() {
  uint64_t x = 88172645463325252ull;  // xorshift64 state
  auto rnd = [&]() { x ^= x << 13; x ^= x >> 7; x ^= x << 17; return x; };
  for (uint32_t d = 1; d <= 3000; ++d) {
    const FastDiv f = make_fastdiv(d);
    for (uint32_t k = 0; k < 64; ++k) {
      const uint64_t base = (uint64_t)d * (k * 1000003u % 70000u);
      for (int e = -1; e <= 1; ++e) {
        const int64_t n = (int64_t)base + e;
        if (n >= 0 && n <= 0xFFFFFFFFll) check((uint32_t)n, d, f);
      }
    }
    check(0u, d, f);
    check(0xFFFFFFFFu, d, f);
    for (int i = 0; i < 200; ++i) check((uint32_t)rnd(), d, f);
  }
  for (int i = 0; i < 20000; ++i) {
    const uint32_t d = (uint32_t)(rnd() % 0x7FFFFFFFull) + 1u;
    const FastDiv f = make_fastdiv(d);
    for (int j = 0; j < 50; ++j) check((uint32_t)rnd(), d, f);
    check(d - 1, d, f); check(d, d, f); check(0xFFFFFFFFu, d, f);
  }
  std::printf(bad ? "FAIL %d\n" : "OK\n", bad);
  return bad ? 1 : 0;
}
"""


def test_fast_division_matches_integer_division(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None or not os.path.isdir(CUDA_INC):
        pytest.skip("needs g++ and the CUDA headers")
    src = tmp_path / "fastdiv.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "fastdiv"
    subprocess.run([cxx, "-std=c++17", "-O2", "-I", CSRC, "-I", CUDA_INC, str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr
