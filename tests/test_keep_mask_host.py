"""Host check of the dropout kernels' keep decision (dropout_keep_msb in the
library's philox.cuh): for every threshold t = 0..255 and every byte value in
every byte position, the top bit of the returned byte must equal byte >= t,
the contract's rule.  Compiled with nvcc as a host program; no GPU needed.
(The GPU probe in test_philox_gpu.py checks the same together with the
byte-to-half-word expansion the kernels apply.)"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_03_gb300", "csrc")

PROGRAM = r"""
#include "philox.cuh"
#include <cstdio>
int main() {
  long long checked = 0;
  for (unsigned t = 0; t < 256; ++t) {
    const unsigned tl4 = (t & 0x7fu) * 0x01010101u, hsel = t >= 128u ? 0xffffffffu : 0u;
    for (unsigned b = 0; b < 256; ++b)
      for (unsigned other = 0; other < 256; other += 17)
        for (int pos = 0; pos < 4; ++pos) {
          // byte b at position pos, the other three bytes varied around it
          unsigned word = 0;
          for (int q = 0; q < 4; ++q) word |= ((q == pos ? b : (other + 61u * q) & 0xffu) << (8 * q));
          const unsigned keep = fa::dropout_keep_msb(word, tl4, hsel);
          for (int q = 0; q < 4; ++q) {
            const unsigned byte = (word >> (8 * q)) & 0xffu;
            if (((keep >> (8 * q + 7)) & 1u) != (byte >= t ? 1u : 0u)) {
              printf("t=%u word=%08x byte %d\n", t, word, q);
              return 1;
            }
            ++checked;
          }
        }
  }
  printf("ok %lld\n", checked);
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc not on PATH")
def test_keep_bits_equal_the_byte_comparison(tmp_path):
    src = tmp_path / "keep.cu"
    exe = tmp_path / "keep"
    src.write_text(PROGRAM)
    subprocess.run(["nvcc", "-std=c++17", "-O2", "-I", CSRC, str(src), "-o", str(exe)],
                   check=True, capture_output=True, timeout=300)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.startswith("ok "), out.stdout + out.stderr
