"""The forward's work-item walk divides by BH, the number of query blocks and
the number of key-range splits with multiply-shift divisors (fa_fastdiv.h).
The header's host path is the same arithmetic as its device path (only the
multiply-high differs: a 64-bit product on the host, __umulhi on the device);
this compiles it with the host compiler and checks it against integer
division: every divisor up to 4096, powers of two and their neighbours, the
largest divisors, and dividends at the edges and spread over 32 bits."""
import os
import shutil
import subprocess

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "exact_attention_98_gb300", "csrc")

PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include "fa_fastdiv.h"
static uint32_t lcg(uint64_t& s) { s = s * 6364136223846793005ull + 1442695040888963407ull; return (uint32_t)(s >> 32); }
static int check(uint32_t d, uint64_t& seed) {
  const fa::FastDiv f(d);
  const uint32_t edge[] = {0u, 1u, d - 1u, d, d + 1u, 2u * d - 1u, 2u * d, 0x7fffffffu, 0x80000000u,
                           0xfffffffeu, 0xffffffffu};
  for (uint32_t n : edge)
    if (f.div(n) != n / d) { printf("d=%u n=%u got %u\n", d, n, f.div(n)); return 1; }
  for (int i = 0; i < 2000; ++i) {
    const uint32_t n = lcg(seed);
    if (f.div(n) != n / d) { printf("d=%u n=%u got %u\n", d, n, f.div(n)); return 1; }
  }
  if (d <= 0x7fffffffu)  // the signed helpers the kernels use (positive int divisors)
    for (int n = 0; n < 3000; ++n)
      if (f.div(n) != n / (int)d || f.mod(n) != n % (int)d) { printf("d=%u n=%d\n", d, n); return 1; }
  return 0;
}
int main() {
  uint64_t seed = 12345;
  for (uint32_t d = 1; d <= 4096; ++d) if (check(d, seed)) return 1;
  for (int k = 1; k < 32; ++k) {
    const uint32_t p = 1u << k;
    if (check(p - 1, seed) || check(p, seed) || (k < 31 && check(p + 1, seed))) return 1;
  }
  if (check(0x7fffffffu, seed) || check(0x80000001u, seed) || check(0xffffffffu, seed)) return 1;
  printf("ok\n");
  return 0;
}
"""


def test_fastdiv_matches_integer_division(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "fastdiv_check.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "fastdiv_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
