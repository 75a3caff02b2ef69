"""Host check of the grid order shared by the prefill and backward kernels
(grouped_tile_order in the library's internal header): for every grid block
it must name one (rank, head) pair, every pair exactly once, and the head
groups must follow the L2 budget rule (l2_head_group).  Compiled with nvcc as
a host program; no GPU needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_03_gb300", "csrc")

PROGRAM = r"""
#include "fa_internal.h"
#include <cstdio>
#include <vector>
int main() {
  const int bhs[] = {1, 3, 7, 8, 9, 16, 31, 64, 67, 512};
  const int nts[] = {1, 2, 3, 16, 64, 65, 256};
  const int groups[] = {1, 2, 5, 8, 12, 64, 1000};
  for (int BH : bhs)
    for (int nt : nts)
      for (int G0 : groups) {
        const int G = G0 > BH ? BH : G0;
        std::vector<int> seen((size_t)BH * nt, 0);
        int prev_group_of_block = -1;
        for (long long b = 0; b < (long long)BH * nt; ++b) {
          const fa::TileOrder t = fa::grouped_tile_order(b, BH, nt, G);
          if (t.rank < 0 || t.rank >= nt || t.bh < 0 || t.bh >= BH) { printf("range %d %d %d\n", BH, nt, G); return 1; }
          if (seen[(size_t)t.bh * nt + t.rank]++) { printf("dup %d %d %d\n", BH, nt, G); return 1; }
          // blocks walk the head groups in order: a block's group never precedes the previous block's
          const int grp = t.bh / G;
          if (grp < prev_group_of_block) { printf("order %d %d %d\n", BH, nt, G); return 1; }
          prev_group_of_block = grp;
        }
      }
  // the budget rule: heads per group = budget / bytes per head, clamped to [1, BH]
  const long long mb = 1ll << 20;
  if (fa::l2_head_group(64, 4 * mb) != 6) { printf("group C3\n"); return 1; }
  if (fa::l2_head_group(32, 32 * mb) != 1) { printf("group C4\n"); return 1; }
  if (fa::l2_head_group(32, 1 * mb) != 24) { printf("group small\n"); return 1; }
  if (fa::l2_head_group(4, 1 * mb) != 4) { printf("group clamp\n"); return 1; }
  printf("ok\n");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc not on PATH")
def test_grouped_tile_order_is_a_bijection(tmp_path):
    src = tmp_path / "order.cu"
    exe = tmp_path / "order"
    src.write_text(PROGRAM)
    subprocess.run(["nvcc", "-std=c++17", "-I", CSRC, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True, timeout=300)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr
