"""CPU check of the multiply-shift division the kernels use for tile and
iteration indices (ra_internal.h: div_magic / div_by).  The header is compiled
as plain host C++ and compared against integer division for every divisor up
to 2^14, on both sides of every multiple and at random points below 2^20."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "blockwise_exact_attention_ra_gb300", "csrc")

PROGRAM = r"""
#include <stdio.h>
#include "ra_internal.h"
int main() {
  unsigned long long checked = 0, rng = 88172645463325252ull;
  for (unsigned d = 1; d <= (1u << 14); ++d) {
    const unsigned long long m = ra::div_magic(d);
    for (unsigned k = 0; (unsigned long long)k * d < (1u << 20); ++k) {
      const int n0 = (int)(k * d);
      const int cand[2] = {n0 - 1, n0};
      for (int c = 0; c < 2; ++c) {
        const int n = cand[c];
        if (n < 0) continue;
        if (ra::div_by(n, m) != n / (int)d) { printf("FAIL %d / %u\n", n, d); return 1; }
        ++checked;
      }
    }
    for (int r = 0; r < 64; ++r) {
      rng ^= rng << 13; rng ^= rng >> 7; rng ^= rng << 17;  // xorshift64
      const int n = (int)(rng & ((1u << 20) - 1));
      if (ra::div_by(n, m) != n / (int)d) { printf("FAIL %d / %u\n", n, d); return 1; }
      ++checked;
    }
  }
  printf("OK %llu\n", checked);
  return 0;
}
"""


def _cuda_include():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime.h")):
            return os.path.join(cand, "include")
    return None


def test_div_by_matches_integer_division(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    inc = _cuda_include()
    if cxx is None or inc is None:
        pytest.skip("needs a host C++ compiler and the CUDA headers")
    src = tmp_path / "div.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "div"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, "-I", inc, str(src), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("OK")
