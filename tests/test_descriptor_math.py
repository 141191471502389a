"""The kernels advance a shared-memory matrix descriptor to the next k-step
with one integer add on its low word (sdesc_add) instead of rebuilding it
from the new address (sdesc_sw128).  The two agree only while the 14-bit
start-address field (address >> 4) does not carry into the next field, that
is while the address stays below 2^18.  This checks, on the host and for
every 1024-byte-aligned tile base below 2^18, every offset form the kernels
use: K-major bf16 k-steps (atoms 8 KB or 16 KB apart, 32 B per step),
MN-major k-steps (2048 B), e4m3 k-steps (32 B).  It also checks that the
largest shared-memory allocation a CTA may have stays below 2^18."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_io_aware_40_gb300", "csrc")

PROGRAM = r"""
#include "ptx.cuh"
#include <cstdio>

int main() {
  using fa::sdesc_add;
  using fa::sdesc_sw128;
  const unsigned kLimit = 1u << 18;
  long checked = 0, bad = 0;
  auto check = [&](unsigned base, unsigned off, unsigned lbo) {
    if (base + off >= kLimit) return;
    ++checked;
    if (sdesc_add(sdesc_sw128(base, lbo, 1024), off) != sdesc_sw128(base + off, lbo, 1024)) {
      if (bad < 5) std::printf("mismatch base %u off %u lbo %u\n", base, off, lbo);
      ++bad;
    }
  };
  for (unsigned base = 0; base < kLimit; base += 1024) {
    for (unsigned atom : {8192u, 16384u})        // K-major bf16, up to d = 256
      for (unsigned k = 0; k < 16; ++k) check(base, (k >> 2) * atom + (k & 3) * 32, 16);
    for (unsigned lbo : {8192u, 16384u})         // MN-major, up to 16 k-steps
      for (unsigned k = 0; k < 16; ++k) check(base, k * 2048, lbo);
    for (unsigned k = 0; k < 4; ++k) check(base, 32 * k, 16);  // e4m3 K-major
  }
  // The largest dynamic + static shared memory a CTA may use on sm_100-class
  // GPUs (227 KB) is below the limit.
  const bool fits = 232448u < kLimit;
  std::printf("%s %ld %ld\n", bad == 0 && fits ? "ok" : "bad", checked, bad);
  return bad == 0 && fits ? 0 : 1;
}
"""


def test_descriptor_advance_matches_rebuild(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("needs nvcc")
    src = tmp_path / "desc.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "desc"
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I" + CSRC, str(src), "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    status, checked, bad = out.stdout.split()[-3:]
    assert status == "ok" and int(bad) == 0 and int(checked) > 10000
